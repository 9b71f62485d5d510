// reconstruct.cu -- the compensated activation of QUADS §3.3, Eq. (21), read back from the
// operand the GEMM consumes (main codes in columns [0, K), the residual tail in [K, K + k)):
//
//   X~[r, j] = DQ(Q(X))[r, j] + DQ(Q(R))[r, p]   when j = S[p] (S the group's channel set)
//   X~[r, j] = DQ(Q(X))[r, j]                    otherwise
//
// with DQ(code) = fl(V * fl(sb * S_dec)) and one binary32 addition.  It is not a step of the
// linear layer: it measures what the compensation buys (the activation error against X).
//
//   dequant_main_kernel   one thread per 16-element block of the main columns: 8 code bytes and
//                         a scale byte in, 16 fp32 values out.
//   add_tail_kernel       one thread per (row, tail column p): the dequantized tail element is
//                         added at channel S[p].  S holds distinct channels, so no two threads of
//                         a row touch the same output; stream order puts it after the first kernel.
#include "common.cuh"

namespace nvq {

static constexpr int kReconThreads = 256;

__global__ void __launch_bounds__(kReconThreads)
    dequant_main_kernel(const uint8_t* __restrict__ codes, int64_t ld_codes, const uint8_t* __restrict__ sf,
                        int64_t sf_cols, const nvq_tensor_scale* __restrict__ ts, Groups gr, int64_t rows,
                        int64_t K, float* __restrict__ out, int64_t ldo)
{
    const int64_t nb = K / 16;
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= rows * nb) return;
    const int64_t r = t / nb, b = t - r * nb;
    const int g = group_of_row(gr, r);
    int64_t g0, g1;
    group_range(gr, g, g0, g1);
    if (r < g0 || r >= g1) return;  // padding row between groups: left as it is
    const float d_b = __fmul_rn(e4m3_value(sf[sf_offset(r, b, sf_cols)]), ts[g].s_dec);
    const uint2 c = *reinterpret_cast<const uint2*>(codes + r * ld_codes + b * 8);
    float v[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t w = (i < 2) ? c.x : c.y;
        const float2 a = e2m1x2_value((w >> (16 * (i & 1))) & 0xffu);
        const float2 a2 = e2m1x2_value((w >> (16 * (i & 1) + 8)) & 0xffu);
        v[4 * i + 0] = __fmul_rn(a.x, d_b);
        v[4 * i + 1] = __fmul_rn(a.y, d_b);
        v[4 * i + 2] = __fmul_rn(a2.x, d_b);
        v[4 * i + 3] = __fmul_rn(a2.y, d_b);
    }
    float4* o = reinterpret_cast<float4*>(out + r * ldo + b * 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

__global__ void __launch_bounds__(kReconThreads)
    add_tail_kernel(const uint8_t* __restrict__ codes, int64_t ld_codes, const uint8_t* __restrict__ sf,
                    int64_t sf_cols, const nvq_tensor_scale* __restrict__ ts, Groups gr, int64_t rows, int64_t K,
                    int k, const int32_t* __restrict__ idx, float* __restrict__ out, int64_t ldo, DeviceStatus* dst)
{
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= rows * k) return;
    const int64_t r = t / k;
    const int p = (int)(t - r * k);
    const int g = group_of_row(gr, r);
    int64_t g0, g1;
    group_range(gr, g, g0, g1);
    if (r < g0 || r >= g1) return;
    const int64_t col = K + p;
    const float d_b = __fmul_rn(e4m3_value(sf[sf_offset(r, col / 16, sf_cols)]), ts[g].s_dec);
    const uint32_t byte = codes[r * ld_codes + col / 2];
    const float2 a = e2m1x2_value(byte);
    const float v = __fmul_rn((p & 1) ? a.y : a.x, d_b);
    float* o = out + r * ldo + checked_channel(idx[(int64_t)g * k + p], (int)K, dst, kWhereBadChannelRecon);
    *o = __fadd_rn(*o, v);
}

}  // namespace nvq

using namespace nvq;

extern "C" nvq_status rac_reconstruct(const uint8_t* codes, int64_t ld_codes, const uint8_t* sf, int64_t sf_cols,
                                      const nvq_tensor_scale* tscale, int64_t rows, int64_t K, int32_t k,
                                      const int32_t* idx, const int64_t* grp_off, const int64_t* grp_rows,
                                      int32_t groups, float* out, int64_t ldo, void* stream)
{
    NVQ_TRACE("rac_reconstruct");
    static const char* fn = "rac_reconstruct";
    NVQ_CHECK_ARG(codes && sf && tscale && out && (k == 0 || idx), NVQ_ERR_ARG, "%s: null pointer", fn);
    NVQ_CHECK_ARG(rows >= 0 && K >= 16 && K % 16 == 0 && groups >= 1, NVQ_ERR_SHAPE,
                  "%s: need rows >= 0, K a positive multiple of 16, groups >= 1", fn);
    NVQ_CHECK_ARG(k >= 0 && k <= K && k % 16 == 0, NVQ_ERR_SHAPE, "%s: k=%d must be a multiple of 16 in [0, K]", fn, k);
    NVQ_CHECK_ARG(ld_codes >= (K + k) / 2 && ldo >= K && sf_cols >= (K + k) / 16, NVQ_ERR_SHAPE,
                  "%s: leading dimension or scale columns too small", fn);
    NVQ_CHECK_ARG(grp_off || rows % groups == 0, NVQ_ERR_SHAPE,
                  "%s: without grp_off the rows split evenly over the groups", fn);
    NVQ_CHECK_ARG(aligned(codes, 8) && ld_codes % 8 == 0 && aligned(out, 16) && ldo % 4 == 0, NVQ_ERR_ALIGN,
                  "%s: codes need 8-byte aligned rows, out 16-byte aligned rows", fn);
    if (rows == 0) return NVQ_OK;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Groups gr{grp_off, grp_rows, groups, rows};
    const int64_t n1 = rows * (K / 16);
    dequant_main_kernel<<<(unsigned)((n1 + kReconThreads - 1) / kReconThreads), kReconThreads, 0, s>>>(
        codes, ld_codes, sf, sf_cols, tscale, gr, rows, K, out, ldo);
    NVQ_LAUNCH_CHECK("rac_reconstruct: dequant_main_kernel");
    if (k > 0) {
        const int64_t n2 = rows * k;
        DeviceStatus* dst = device_status_ptr();
        NVQ_CHECK_ARG(dst, NVQ_ERR_CUDA, "%s: device status word unavailable", fn);
        add_tail_kernel<<<(unsigned)((n2 + kReconThreads - 1) / kReconThreads), kReconThreads, 0, s>>>(
            codes, ld_codes, sf, sf_cols, tscale, gr, rows, K, k, idx, out, ldo, dst);
        NVQ_LAUNCH_CHECK("rac_reconstruct: add_tail_kernel");
    }
    return NVQ_OK;
}
