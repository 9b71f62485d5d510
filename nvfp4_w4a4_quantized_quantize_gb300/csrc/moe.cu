// moe.cu -- routing plumbing around the grouped W4A4 GEMM of the MoE expert layer.
//
// The paper runs its RAC linear layers inside the experts of an MoE model (QUADS §3.3, the
// "W13" activation site; §4.1 MoE 25B-A2.8B) but does not describe dispatch or combine; these
// are the plain steps of a top-k routed layer:
//   dispatch   stable counting sort of the (token, slot) pairs by expert; every expert's rows
//              start on a multiple of 128 so that a 128-row GEMM tile never spans two experts
//              and the blocked scale layout stays tile-aligned;
//   gather     copies each routed row's quantized codes and scales from its token row (NVFP4
//              rows, with their RAC tail, or the FP8 baseline's rows);
//   combine    sums each token's topk expert outputs in slot order (fp32) and rounds to bf16.
#include <cuda_bf16.h>

#include <mutex>

#include "common.cuh"

namespace nvq {

// Pairs are cut into units of 256 consecutive (token, slot) pairs; one warp owns a unit.
static constexpr int kUnit = 256;
static constexpr int kWarpsPerCta = 2;  // 256 CTAs for the 512 units of 131072 pairs: every SM busy

// An expert id outside [0, G) is a caller error: the pair is left out of the routing (its
// row_of entry is -1, which combine skips) and the device status word records NVQ_ERR_ARG.
static constexpr int kWhereBadExpertId = 41;
static constexpr int kWhereBadSourceRow = 45;  // gather: row_src[i] / topk >= src_rows

// Per-unit histogram of experts: counts[unit][G].
__global__ void dispatch_hist_kernel(const int32_t* __restrict__ ids, int64_t n, int G, int32_t* __restrict__ counts,
                                     DeviceStatus* __restrict__ st)
{
    extern __shared__ int32_t hist[];  // [kWarpsPerCta][G]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int32_t* h = hist + warp * G;
    for (int e = lane; e < G; e += 32) h[e] = 0;
    __syncwarp();
    const int64_t unit = (int64_t)blockIdx.x * kWarpsPerCta + warp;
    const int64_t p0 = unit * kUnit;
    if (p0 >= n) return;
    const int64_t p1 = min(p0 + kUnit, n);
    for (int64_t p = p0 + lane; p < p1; p += 32) {
        const int e = ids[p];
        if ((unsigned)e < (unsigned)G) atomicAdd(&h[e], 1);
        else report_status(st, NVQ_ERR_ARG, kWhereBadExpertId);
    }
    __syncwarp();
    for (int e = lane; e < G; e += 32) counts[unit * G + e] = h[e];
}

// CTA per expert: exclusive scan of its count over units; grp_rows[e] = total.
__global__ void __launch_bounds__(1024) dispatch_scan_kernel(int32_t* __restrict__ counts, int units, int G,
                                                             int64_t* __restrict__ grp_rows)
{
    __shared__ int warp_sums[32];
    const int e = blockIdx.x;
    const int per = (units + blockDim.x - 1) / blockDim.x;
    const int u0 = threadIdx.x * per, u1 = min(units, u0 + per);
    int local = 0;
    for (int u = u0; u < u1; ++u) local += counts[(int64_t)u * G + e];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int s = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        warp_sums[lane] = s;
    }
    __syncthreads();
    int run = (warp ? warp_sums[warp - 1] : 0) + x - local;
    for (int u = u0; u < u1; ++u) {
        int v = counts[(int64_t)u * G + e];
        counts[(int64_t)u * G + e] = run;
        run += v;
    }
    if (threadIdx.x == blockDim.x - 1) grp_rows[e] = run;
}

// One CTA of 1024 threads: 128-padded group offsets (block scan) and the padding rows.
__global__ void __launch_bounds__(1024) dispatch_offsets_kernel(int G, const int64_t* __restrict__ grp_rows,
                                                                int64_t* __restrict__ grp_off, int32_t* __restrict__ row_src,
                                                                float* __restrict__ row_w, int64_t capacity)
{
    __shared__ int64_t warp_sums[32];
    __shared__ int64_t off[1025];
    const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
    const int64_t padded = e < G ? (grp_rows[e] + 127) / 128 * 128 : 0;
    int64_t x = padded;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int64_t w = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    const int64_t excl = (warp ? warp_sums[warp - 1] : 0) + x - padded;
    if (e < G) off[e] = excl;
    if (e == G - 1) off[G] = excl + padded;
    __syncthreads();
    if (e <= G) grp_off[e] = off[e];
    // padding rows: inside each group after its routed rows, then up to the capacity
    const int64_t total = off[G];
    for (int g = warp; g < G; g += 32) {
        const int64_t end = off[g] + grp_rows[g];
        for (int64_t r = end + lane; r < off[g + 1]; r += 32) {
            row_src[r] = -1;
            if (row_w) row_w[r] = 0.0f;
        }
    }
    for (int64_t r = total + e; r < capacity; r += 1024) {
        row_src[r] = -1;
        if (row_w) row_w[r] = 0.0f;
    }
}

// Warp per unit keeps the (token, slot) order inside every expert.
__global__ void dispatch_scatter_kernel(const int32_t* __restrict__ ids, const float* __restrict__ w, int64_t n, int G,
                                        const int32_t* __restrict__ counts, const int64_t* __restrict__ grp_off,
                                        int32_t* __restrict__ row_src, int64_t* __restrict__ row_of,
                                        float* __restrict__ row_w)
{
    extern __shared__ int64_t base_all[];  // [kWarpsPerCta][G]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int64_t* base = base_all + warp * G;
    const int64_t unit = (int64_t)blockIdx.x * kWarpsPerCta + warp;
    const int64_t p0 = unit * kUnit;
    if (p0 >= n) return;
    for (int e = lane; e < G; e += 32) base[e] = grp_off[e] + counts[unit * G + e];
    __syncwarp();
    const int64_t p1 = min(p0 + kUnit, n);
    // the unit's expert ids and weights, all loads in flight before the ranking
    constexpr int kPer = kUnit / 32;
    int ev[kPer];
    float wv[kPer];
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        const int64_t p = p0 + q * 32 + lane;
        ev[q] = p < p1 ? ids[p] : 0;
        wv[q] = (p < p1 && w) ? w[p] : 1.0f;
    }
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        const int64_t p = p0 + q * 32 + lane;
        const bool in_id = (unsigned)ev[q] < (unsigned)G;  // the histogram kernel reported the others
        if (p < p1 && !in_id) row_of[p] = -1;
        const bool valid = p < p1 && in_id;
        const unsigned act = __ballot_sync(0xffffffffu, valid);
        const int e = ev[q];
        int rank = 0;
        unsigned peers = 0;
        if (valid) {
            peers = __match_any_sync(act, e);
            rank = __popc(peers & ((1u << lane) - 1u));
            const int64_t pos = base[e] + rank;
            row_src[pos] = (int32_t)p;
            row_of[p] = pos;
            if (row_w) row_w[pos] = wv[q];
        }
        __syncwarp();
        if (valid && rank == 0) base[e] += __popc(peers);
        __syncwarp();
    }
}

// CTA (or gridDim.y CTAs, splitting its bytes, when there are few blocks) per 128-row block of
// the routed layout.  Codes: bytes [byte0, byte_end) of every row,
// 16-byte vectors (an 8-byte piece at the end when byte_end % 16 == 8).  Scales: the 512-byte
// atoms [atom0, atom_end) of the row block (4 scale columns each), the block's output words
// written in the blocked layout's own order (coalesced); each reads its word from the source
// row's scales (token scales: small and L2 resident).  NVFP4 rows of ktot elements hold ktot / 2
// code bytes and ktot / 64 atoms; FP8 rows of K elements hold K bytes and K / 128 atoms.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint8_t* __restrict__ codes, int64_t ld_codes,
                                                          const uint8_t* __restrict__ sf, int64_t sf_cols,
                                                          const int32_t* __restrict__ row_src, int topk, int64_t byte0,
                                                          int64_t byte_end, int atom0, int atom_end,
                                                          uint8_t* __restrict__ out_codes, int64_t ld_out,
                                                          uint8_t* __restrict__ out_sf, int64_t src_rows, DeviceStatus* dst)
{
    __shared__ int src[128];
    const int tid = threadIdx.x;
    const int64_t r0 = (int64_t)blockIdx.x * 128;
    if (tid < 128) {
        const int32_t s = row_src[r0 + tid];
        int v = s >= 0 ? s / topk : -1;
        if (v >= src_rows) {  // a row map not made for this source: recorded, and the row is left as padding
            report_status(dst, NVQ_ERR_ARG, kWhereBadSourceRow);
            v = -1;
        }
        src[tid] = v;
    }
    __syncthreads();
    if (out_codes != nullptr) {
        // the block's 128 rows x nv 16-byte vectors as one flat range, consecutive threads on
        // consecutive vectors of a row: every lane busy, eight loads in flight per thread before
        // their stores
        const int v_begin = (int)(byte0 / 16);
        const int nv = (int)(byte_end / 16) - v_begin;  // 16-byte vectors per row
        const int total = 128 * nv;
        // this CTA's share of the block (gridDim.y CTAs per block when blocks are few)
        const int chunk = (total + (int)gridDim.y - 1) / (int)gridDim.y;
        const int lo = (int)blockIdx.y * chunk, hi = min(total, lo + chunk);
        for (int i0 = lo + tid; i0 < hi; i0 += 8 * 256) {
            uint4 val[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = i0 + j * 256;
                val[j] = make_uint4(0, 0, 0, 0);
                if (i < hi) {
                    const int r = i / nv, v = v_begin + (i - r * nv);
                    const int sr = src[r];
                    if (sr >= 0) val[j] = __ldg(reinterpret_cast<const uint4*>(codes + (int64_t)sr * ld_codes) + v);
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = i0 + j * 256;
                if (i < hi) {
                    const int r = i / nv, v = v_begin + (i - r * nv);
                    reinterpret_cast<uint4*>(out_codes + (r0 + r) * ld_out)[v] = val[j];
                }
            }
        }
        if ((byte_end % 16) != 0 && blockIdx.y == 0 && tid < 128) {  // the 8-byte piece at the end of each row
            const int64_t off = byte_end - 8;
            const int sr = src[tid];
            *reinterpret_cast<uint2*>(out_codes + (r0 + tid) * ld_out + off) =
                sr >= 0 ? *reinterpret_cast<const uint2*>(codes + (int64_t)sr * ld_codes + off) : make_uint2(0, 0);
        }
    }
    // scales: four words per thread at a time, loads before stores
    const int natoms = (int)(sf_cols / 4);
    const int wchunk = (atom_end * 128 - atom0 * 128 + (int)gridDim.y - 1) / (int)gridDim.y;
    const int wlo = atom0 * 128 + (int)blockIdx.y * wchunk;
    const int nwords = min(atom_end * 128, wlo + wchunk);  // this CTA's words end here
    uint32_t* outw = reinterpret_cast<uint32_t*>(out_sf + blockIdx.x * (int64_t)natoms * 512);
    for (int w0 = wlo + tid; w0 < nwords; w0 += 4 * 256) {
        uint32_t val[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int w = w0 + i * 256;
            val[i] = 0u;
            if (w < nwords) {
                const int a = w >> 7, pos = w & 127;
                const int r = (pos >> 2) + 32 * (pos & 3);
                const int sr = src[r];
                if (sr >= 0) val[i] = __ldg(reinterpret_cast<const uint32_t*>(sf + sf_offset(sr, 4 * a, sf_cols)));
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (w0 + i * 256 < nwords) outw[w0 + i * 256] = val[i];
    }
}

// CTA per token; each thread sums 8 columns over the slots in slot order.  The token's slot rows
// are read once into shared memory; for up to kCombineSlots slots every thread then has all its
// loads in flight before the first add (a runtime-bounded loop would wait on each slot's load
// in turn).  Larger topk takes the same sum slot by slot.
constexpr int kCombineSlots = 8;

__device__ __forceinline__ void add_bf16x8(float* acc, const uint4& w)
{
    acc[0] = __fadd_rn(acc[0], bf16lo(w.x)); acc[1] = __fadd_rn(acc[1], bf16hi(w.x));
    acc[2] = __fadd_rn(acc[2], bf16lo(w.y)); acc[3] = __fadd_rn(acc[3], bf16hi(w.y));
    acc[4] = __fadd_rn(acc[4], bf16lo(w.z)); acc[5] = __fadd_rn(acc[5], bf16hi(w.z));
    acc[6] = __fadd_rn(acc[6], bf16lo(w.w)); acc[7] = __fadd_rn(acc[7], bf16hi(w.w));
}

__global__ void combine_kernel(const __nv_bfloat16* __restrict__ y, int64_t ldy, const int64_t* __restrict__ row_of,
                               int topk, int64_t hidden, __nv_bfloat16* __restrict__ out, int64_t ldo)
{
    __shared__ int64_t s_row[kCombineSlots];
    const int64_t t = blockIdx.x;
    const bool few = topk <= kCombineSlots;
    if (few && threadIdx.x < topk) s_row[threadIdx.x] = row_of[t * topk + threadIdx.x];
    __syncthreads();
    for (int64_t c = (int64_t)threadIdx.x * 8; c < hidden; c += (int64_t)blockDim.x * 8) {
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        if (few) {
            uint4 w[kCombineSlots];
#pragma unroll
            for (int s = 0; s < kCombineSlots; ++s) {
                const int64_t r = s < topk ? s_row[s] : -1;
                w[s] = r >= 0 ? __ldg(reinterpret_cast<const uint4*>(y + r * ldy + c)) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int s = 0; s < kCombineSlots; ++s)
                if (s < topk && s_row[s] >= 0) add_bf16x8(acc, w[s]);  // slot order; a pair left out adds nothing
        } else {
            for (int s = 0; s < topk; ++s) {
                const int64_t r = row_of[t * topk + s];
                if (r < 0) continue;  // a pair dispatch left out (expert id out of range)
                add_bf16x8(acc, __ldg(reinterpret_cast<const uint4*>(y + r * ldy + c)));
            }
        }
        uint32_t pk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
            pk[i] = *reinterpret_cast<uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(out + t * ldo + c) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
}

// One CTA per 128-row block, or up to 8 per block (splitting its bytes) until there are about
// four CTAs per SM: the decode shapes have few blocks (capacity 20352 rows: 159 blocks).
static dim3 gather_grid(int64_t capacity)
{
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t blocks = capacity / 128;
    int64_t split = (4 * (int64_t)sms + blocks - 1) / blocks;
    if (split < 1) split = 1;
    if (split > 8) split = 8;
    return dim3((unsigned)blocks, (unsigned)split);
}

}  // namespace nvq

using namespace nvq;

extern "C" int64_t moe_capacity(int64_t tokens, int32_t topk, int32_t groups)
{
    return (tokens * topk + 127) / 128 * 128 + (int64_t)groups * 128;
}

extern "C" size_t moe_dispatch_workspace_size(int64_t tokens, int32_t topk, int32_t groups)
{
    const int64_t units = (tokens * topk + kUnit - 1) / kUnit;
    return (size_t)(units * groups * sizeof(int32_t));
}

extern "C" nvq_status moe_dispatch(const int32_t* topk_ids, const float* topk_w, int64_t tokens, int32_t topk,
                                   int32_t groups, int64_t* grp_off, int64_t* grp_rows, int32_t* row_src,
                                   int64_t* row_of, float* row_w, int64_t capacity, void* workspace,
                                   size_t workspace_bytes, void* stream)
{
    NVQ_TRACE("moe_dispatch");
    NVQ_CHECK_ARG(topk_ids && grp_off && grp_rows && row_src && row_of && workspace, NVQ_ERR_ARG,
                  "moe_dispatch: null pointer argument");
    NVQ_CHECK_ARG(tokens >= 1 && topk >= 1 && topk <= 64 && tokens * topk <= (1ll << 26), NVQ_ERR_SHAPE,
                  "moe_dispatch: tokens*topk outside [1, 2^26] or topk outside [1, 64]");
    NVQ_CHECK_ARG(groups >= 1 && groups <= 1024, NVQ_ERR_SHAPE, "moe_dispatch: groups outside [1, 1024]");
    NVQ_CHECK_ARG(capacity >= moe_capacity(tokens, topk, groups), NVQ_ERR_SHAPE,
                  "moe_dispatch: capacity %lld < moe_capacity() = %lld", (long long)capacity,
                  (long long)moe_capacity(tokens, topk, groups));
    NVQ_CHECK_ARG(workspace_bytes >= moe_dispatch_workspace_size(tokens, topk, groups), NVQ_ERR_SHAPE,
                  "moe_dispatch: workspace too small");
    DeviceStatus* dstat = device_status_ptr();
    NVQ_CHECK_ARG(dstat, NVQ_ERR_CUDA, "moe_dispatch: device status word unavailable");
    set_error("");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t n = tokens * topk;
    const int units = (int)((n + kUnit - 1) / kUnit);
    const int ctas = (units + kWarpsPerCta - 1) / kWarpsPerCta;
    int32_t* counts = static_cast<int32_t*>(workspace);
    dispatch_hist_kernel<<<ctas, 32 * kWarpsPerCta, kWarpsPerCta * groups * sizeof(int32_t), st>>>(topk_ids, n, groups, counts,
                                                                                                   dstat);
    NVQ_LAUNCH_CHECK("dispatch_hist_kernel");
    dispatch_scan_kernel<<<groups, units >= 1024 ? 1024 : ((units + 31) / 32) * 32, 0, st>>>(counts, units, groups, grp_rows);
    NVQ_LAUNCH_CHECK("dispatch_scan_kernel");
    dispatch_offsets_kernel<<<1, 1024, 0, st>>>(groups, grp_rows, grp_off, row_src, row_w, capacity);
    NVQ_LAUNCH_CHECK("dispatch_offsets_kernel");
    dispatch_scatter_kernel<<<ctas, 32 * kWarpsPerCta, kWarpsPerCta * groups * sizeof(int64_t), st>>>(
        topk_ids, topk_w, n, groups, counts, grp_off, row_src, row_of, row_w);
    NVQ_LAUNCH_CHECK("dispatch_scatter_kernel");
    return NVQ_OK;
}

extern "C" nvq_status nvfp4_gather_rows(const uint8_t* codes, int64_t ld_codes, const uint8_t* sf, int64_t sf_cols,
                                        int64_t src_rows, const int32_t* row_src, int32_t topk, int64_t capacity,
                                        int64_t ktot, int64_t col0, uint8_t* out_codes, int64_t ld_out, uint8_t* out_sf,
                                        void* stream)
{
    NVQ_TRACE("nvfp4_gather_rows");
    NVQ_CHECK_ARG(codes && sf && row_src && out_sf, NVQ_ERR_ARG, "nvfp4_gather_rows: null pointer argument");
    NVQ_CHECK_ARG(ktot >= 16 && ktot % 16 == 0 && sf_cols >= ktot / 16 && sf_cols % 4 == 0, NVQ_ERR_SHAPE,
                  "nvfp4_gather_rows: bad ktot / sf_cols");
    NVQ_CHECK_ARG(capacity >= 1 && capacity % 128 == 0 && src_rows >= 1 && topk >= 1, NVQ_ERR_SHAPE,
                  "nvfp4_gather_rows: capacity must be a positive multiple of 128");
    NVQ_CHECK_ARG(col0 >= 0 && col0 % 64 == 0 && col0 < ktot, NVQ_ERR_SHAPE,
                  "nvfp4_gather_rows: col0 must be a multiple of 64 below ktot");
    NVQ_CHECK_ARG(ld_codes % 16 == 0 && ld_codes >= ktot / 2 && aligned(codes, 16) && aligned(sf, 4) && aligned(out_sf, 4) &&
                      (!out_codes || (ld_out % 16 == 0 && ld_out >= ktot / 2 && aligned(out_codes, 16))),
                  NVQ_ERR_ALIGN, "nvfp4_gather_rows: codes need 16-byte aligned rows");
    set_error("");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    DeviceStatus* dst = device_status_ptr();
    NVQ_CHECK_ARG(dst, NVQ_ERR_CUDA, "nvfp4_gather_rows: device status word unavailable");
    gather_rows_kernel<<<gather_grid(capacity), 256, 0, st>>>(codes, ld_codes, sf, sf_cols, row_src, topk, col0 / 2,
                                                                   ktot / 2, (int)(col0 / 64), (int)((ktot + 63) / 64),
                                                                   out_codes, ld_out, out_sf, src_rows, dst);
    NVQ_LAUNCH_CHECK("gather_rows_kernel");
    return NVQ_OK;
}

extern "C" nvq_status fp8_gather_rows(const uint8_t* codes, int64_t ld_codes, const uint8_t* sf, int64_t sf_cols,
                                      int64_t src_rows, const int32_t* row_src, int32_t topk, int64_t capacity, int64_t K,
                                      uint8_t* out_codes, int64_t ld_out, uint8_t* out_sf, void* stream)
{
    NVQ_TRACE("fp8_gather_rows");
    NVQ_CHECK_ARG(codes && sf && row_src && out_codes && out_sf, NVQ_ERR_ARG, "fp8_gather_rows: null pointer argument");
    NVQ_CHECK_ARG(K >= 32 && K % 32 == 0 && sf_cols >= nvq_fp8_sf_cols(K) && sf_cols % 4 == 0, NVQ_ERR_SHAPE,
                  "fp8_gather_rows: K must be a positive multiple of 32 and sf_cols >= nvq_fp8_sf_cols(K)");
    NVQ_CHECK_ARG(capacity >= 1 && capacity % 128 == 0 && src_rows >= 1 && topk >= 1, NVQ_ERR_SHAPE,
                  "fp8_gather_rows: capacity must be a positive multiple of 128");
    NVQ_CHECK_ARG(ld_codes % 16 == 0 && ld_codes >= K && aligned(codes, 16) && aligned(sf, 4) && aligned(out_sf, 4) &&
                      ld_out % 16 == 0 && ld_out >= K && aligned(out_codes, 16),
                  NVQ_ERR_ALIGN, "fp8_gather_rows: codes need 16-byte aligned rows");
    set_error("");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    DeviceStatus* dst = device_status_ptr();
    NVQ_CHECK_ARG(dst, NVQ_ERR_CUDA, "fp8_gather_rows: device status word unavailable");
    gather_rows_kernel<<<gather_grid(capacity), 256, 0, st>>>(codes, ld_codes, sf, sf_cols, row_src, topk, 0, K, 0,
                                                                   (int)((K + 127) / 128), out_codes, ld_out, out_sf,
                                                                   src_rows, dst);
    NVQ_LAUNCH_CHECK("gather_rows_kernel");
    return NVQ_OK;
}

extern "C" nvq_status moe_combine(const void* y, int64_t ldy, const int64_t* row_of, int64_t tokens, int32_t topk,
                                  int64_t hidden, void* out, int64_t ldo, void* stream)
{
    NVQ_TRACE("moe_combine");
    NVQ_CHECK_ARG(y && row_of && out, NVQ_ERR_ARG, "moe_combine: null pointer argument");
    NVQ_CHECK_ARG(tokens >= 1 && tokens <= (1ll << 31) - 1 && topk >= 1 && hidden >= 8 && hidden % 8 == 0, NVQ_ERR_SHAPE,
                  "moe_combine: hidden must be a positive multiple of 8");
    NVQ_CHECK_ARG(ldy % 8 == 0 && ldo % 8 == 0 && ldy >= hidden && ldo >= hidden && aligned(y, 16) && aligned(out, 16),
                  NVQ_ERR_ALIGN, "moe_combine: rows must be 16-byte aligned");
    set_error("");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    combine_kernel<<<(unsigned)tokens, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(y), ldy, row_of, topk, hidden,
                                                     static_cast<__nv_bfloat16*>(out), ldo);
    NVQ_LAUNCH_CHECK("combine_kernel");
    return NVQ_OK;
}

// ------------------------------------------------------------------------ dispatch, static scratch
// moe_dispatch_static_scratch: the same four kernels as moe_dispatch, with the per-unit expert
// histogram (counts[units][groups], int32) kept in one file-scope device array instead of a
// caller workspace, so that the call allocates nothing.  Its address is looked up once per device
// (first call on that device, with the device current) and cached.
namespace nvq {

static constexpr size_t kDispatchScratchBytes = NVQ_DISPATCH_STATIC_SCRATCH_BYTES;
static constexpr int kScratchMaxDevices = 64;

static __device__ __align__(256) int32_t g_dispatch_scratch[kDispatchScratchBytes / sizeof(int32_t)];

static std::mutex g_scratch_mu;
static void* g_scratch_addr[kScratchMaxDevices];

// Device address of g_dispatch_scratch on the current device (set-up on the first call).
static nvq_status dispatch_scratch_ptr(int32_t** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e, "moe_dispatch_static_scratch: cudaGetDevice");
    if (dev < 0 || dev >= kScratchMaxDevices) {
        set_error("moe_dispatch_static_scratch: device ordinal %d outside [0, %d)", dev, kScratchMaxDevices);
        return NVQ_ERR_ARG;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
        if (e != cudaSuccess) return cuda_status(e, "moe_dispatch_static_scratch: cudaGetSymbolAddress(g_dispatch_scratch)");
        g_scratch_addr[dev] = p;
    }
    *out = static_cast<int32_t*>(g_scratch_addr[dev]);
    return NVQ_OK;
}

}  // namespace nvq

extern "C" nvq_status moe_dispatch_static_scratch(const int32_t* topk_ids, const float* topk_w, int64_t tokens,
                                                  int32_t topk, int32_t groups, int64_t* grp_off, int64_t* grp_rows,
                                                  int32_t* row_src, int64_t* row_of, float* row_w, int64_t capacity,
                                                  void* stream)
{
    NVQ_TRACE("moe_dispatch_static_scratch");
    NVQ_CHECK_ARG(topk_ids && grp_off && grp_rows && row_src && row_of, NVQ_ERR_ARG,
                  "moe_dispatch_static_scratch: null pointer argument");
    NVQ_CHECK_ARG(tokens >= 1 && topk >= 1 && topk <= 64 && tokens * topk <= (1ll << 26), NVQ_ERR_SHAPE,
                  "moe_dispatch_static_scratch: tokens*topk outside [1, 2^26] or topk outside [1, 64]");
    // the same group limit as moe_dispatch: the scatter kernel's shared table of group bases
    // (kWarpsPerCta x groups x 8 bytes, 16 KB at 1024 groups) stays within the 48 KB a launch
    // gets without an attribute call
    NVQ_CHECK_ARG(groups >= 1 && groups <= 1024, NVQ_ERR_SHAPE, "moe_dispatch_static_scratch: groups outside [1, 1024]");
    NVQ_CHECK_ARG(capacity >= moe_capacity(tokens, topk, groups), NVQ_ERR_SHAPE,
                  "moe_dispatch_static_scratch: capacity %lld < moe_capacity() = %lld", (long long)capacity,
                  (long long)moe_capacity(tokens, topk, groups));
    const size_t need = moe_dispatch_workspace_size(tokens, topk, groups);
    NVQ_CHECK_ARG(need <= kDispatchScratchBytes, NVQ_ERR_SHAPE,
                  "moe_dispatch_static_scratch: tokens=%lld topk=%d groups=%d need %zu bytes of scratch, more than the "
                  "%zu-byte static array; call moe_dispatch with a workspace instead",
                  (long long)tokens, (int)topk, (int)groups, need, kDispatchScratchBytes);
    int32_t* counts = nullptr;
    const nvq_status s = dispatch_scratch_ptr(&counts);
    if (s != NVQ_OK) return s;
    DeviceStatus* dstat = device_status_ptr();
    NVQ_CHECK_ARG(dstat, NVQ_ERR_CUDA, "moe_dispatch_static_scratch: device status word unavailable");
    set_error("");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t n = tokens * topk;
    const int units = (int)((n + kUnit - 1) / kUnit);
    const int ctas = (units + kWarpsPerCta - 1) / kWarpsPerCta;
    // every counts word the later kernels read is written by the histogram kernel of this call:
    // nothing in the scratch has to start at zero
    dispatch_hist_kernel<<<ctas, 32 * kWarpsPerCta, kWarpsPerCta * groups * sizeof(int32_t), st>>>(topk_ids, n, groups, counts,
                                                                                                   dstat);
    NVQ_LAUNCH_CHECK("dispatch_hist_kernel");
    dispatch_scan_kernel<<<groups, units >= 1024 ? 1024 : ((units + 31) / 32) * 32, 0, st>>>(counts, units, groups, grp_rows);
    NVQ_LAUNCH_CHECK("dispatch_scan_kernel");
    dispatch_offsets_kernel<<<1, 1024, 0, st>>>(groups, grp_rows, grp_off, row_src, row_w, capacity);
    NVQ_LAUNCH_CHECK("dispatch_offsets_kernel");
    dispatch_scatter_kernel<<<ctas, 32 * kWarpsPerCta, kWarpsPerCta * groups * sizeof(int64_t), st>>>(
        topk_ids, topk_w, n, groups, counts, grp_off, row_src, row_of, row_w);
    NVQ_LAUNCH_CHECK("dispatch_scatter_kernel");
    return NVQ_OK;
}
