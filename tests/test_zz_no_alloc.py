"""moe_dispatch_static_scratch, the dispatch entry that allocates nothing, checked against
moe_dispatch (caller workspace) on the same routing: two calls in a row with different sizes,
so the second call runs over scratch the first one left behind, then a request larger than the
static array, which must be refused before any launch.  Collected last so that it also runs
after every other test in the same process; it passes alone as well."""
import numpy as np
import pytest
import torch

from nvfp4_w4a4_quantized_quantize_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from nvfp4_w4a4_quantized_quantize_gb300 import _lib
    return _lib


def _outputs(L, T, topk, E, cap, dev):
    return dict(grp_off=torch.full((E + 1,), -7, dtype=torch.int64, device=dev),
                grp_rows=torch.full((E,), -7, dtype=torch.int64, device=dev),
                row_src=torch.full((cap,), -7, dtype=torch.int32, device=dev),
                row_of=torch.full((T * topk,), -7, dtype=torch.int64, device=dev),
                row_w=torch.full((cap,), -7.0, dtype=torch.float32, device=dev))


def _both(L, ids_np, w_np, E):
    dev = "cuda"
    T, topk = ids_np.shape
    ids = torch.from_numpy(ids_np).to(dev)
    w = torch.from_numpy(w_np).to(dev)
    cap = L.moe_capacity(T, topk, E)
    ref = _outputs(L, T, topk, E, cap, dev)
    ws = torch.zeros(L.moe_dispatch_workspace_size(T, topk, E), dtype=torch.uint8, device=dev)
    L.moe_dispatch(ids, w, E, ref["grp_off"], ref["grp_rows"], ref["row_src"], ref["row_of"], ref["row_w"], ws)
    got = _outputs(L, T, topk, E, cap, dev)
    L.moe_dispatch_static_scratch(ids, w, E, got["grp_off"], got["grp_rows"], got["row_src"], got["row_of"],
                                  got["row_w"])
    torch.cuda.synchronize()
    return ref, got


def _assert_same(ref, got):
    # integer outputs bit-exact; the routing weights are copied, so exact as well
    for name in ("grp_off", "grp_rows", "row_src", "row_of"):
        assert torch.equal(ref[name], got[name]), name
    assert torch.equal(ref["row_w"].view(torch.int32), got["row_w"].view(torch.int32))


def test_static_scratch_dispatch_matches_workspace_dispatch_twice(L):
    # call 1: the prefill routing at 8192 tokens (Zipf, 128 experts, top-8): 256 units of 256
    # (token, slot) pairs x 128 experts x 4 bytes = 128 KiB of scratch
    ids1, w1 = wl.routing_zipf(8192, 128, 8, 1.1, seed=31)
    ref1, got1 = _both(L, ids1, w1, 128)
    _assert_same(ref1, got1)
    # call 2, right after: a smaller uniform routing over 8 experts reuses the same array
    ids2, w2 = wl.routing_uniform(300, 8, 2, seed=32)
    ref2, got2 = _both(L, ids2, w2, 8)
    _assert_same(ref2, got2)
    # sanity of the shared result (the workspace entry is itself checked against the oracle elsewhere)
    counts = np.bincount(ids2.ravel(), minlength=8)
    assert np.array_equal(got2["grp_rows"].cpu().numpy(), counts)


def test_static_scratch_dispatch_refuses_oversize(L):
    T, topk, E = 70000, 8, 128  # 2188 units x 128 experts x 4 bytes > 1 MiB
    assert L.moe_dispatch_workspace_size(T, topk, E) > (1 << 20)
    dev = "cuda"
    ids = torch.zeros(T, topk, dtype=torch.int32, device=dev)
    out = _outputs(L, T, topk, E, L.moe_capacity(T, topk, E), dev)
    with pytest.raises(L.NvqError) as ei:
        L.moe_dispatch_static_scratch(ids, None, E, out["grp_off"], out["grp_rows"], out["row_src"], out["row_of"],
                                      out["row_w"])
    assert ei.value.status == 2 and "static array" in str(ei.value)
    torch.cuda.synchronize()
    assert int(out["grp_off"][0]) == -7  # nothing was launched


def test_static_scratch_dispatch_at_exactly_the_limit(L):
    # 65536 tokens at top-8 over 128 experts: 2048 units x 128 x 4 bytes = 1 MiB, the whole array
    T, topk, E = 65536, 8, 128
    assert L.moe_dispatch_workspace_size(T, topk, E) == (1 << 20)
    ids, w = wl.routing_zipf(T, E, topk, 1.1, seed=33)
    ref, got = _both(L, ids, w, E)
    _assert_same(ref, got)
    assert np.array_equal(got["grp_rows"].cpu().numpy(), np.bincount(ids.ravel(), minlength=E))


def test_static_scratch_dispatch_refuses_too_many_groups(L):
    T, topk, E = 64, 2, 1025  # one group more than moe_dispatch accepts
    dev = "cuda"
    ids = torch.zeros(T, topk, dtype=torch.int32, device=dev)
    out = _outputs(L, T, topk, E, L.moe_capacity(T, topk, E), dev)
    with pytest.raises(L.NvqError) as ei:
        L.moe_dispatch_static_scratch(ids, None, E, out["grp_off"], out["grp_rows"], out["row_src"], out["row_of"],
                                      out["row_w"])
    assert ei.value.status == 2 and "groups" in str(ei.value)
    torch.cuda.synchronize()
    assert int(out["grp_off"][0]) == -7  # nothing was launched
