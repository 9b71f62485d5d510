// quantize.cu -- NVFP4 quantization of bf16 matrices (QUADS §2.2 "FP4"; Q_A of Eq. (9),
// Q_W of Eq. (7) and the trainer's QDQ_W of Eq. (12)) with the per-channel residual score of
// Eq. (23) fused into the same pass over the input.
//
// Two kernels per call:
//   amax_kernel          per-group max |x| (the FP32 tensor scale's statistic), one atomicMax
//                        per (CTA, group run);
//   quant_score_kernel   codes + blocked E4M3 scales + residual + integer channel score (+ the
//                        dequantized values for the trainer-side QDQ), one thread per
//                        16-element block, 32-byte coalesced loads.
// Both are HBM-bound: the input is read twice (the second read is mostly served by L2 for
// inputs up to ~100 MB), codes and scales are written once.
#include <cuda_bf16.h>

#include "common.cuh"

namespace nvq {

static constexpr int kQuantThreads = 256;

// ------------------------------------------------------------------------ amax
__global__ void __launch_bounds__(kQuantThreads) amax_kernel(const __nv_bfloat16* __restrict__ x, int64_t ldx,
                                                              int K, Groups gr, int64_t rows_per_cta,
                                                              nvq_tensor_scale* __restrict__ ts)
{
    __shared__ float red[kQuantThreads / 32];
    const int64_t r0 = (int64_t)blockIdx.x * rows_per_cta;
    const int64_t r1 = min(r0 + rows_per_cta, gr.total_rows);
    if (r0 >= r1) return;
    const int vec_per_row = K / 8;
    int g = group_of_row(gr, r0);
    int64_t row = r0;
    while (row < r1 && g < gr.G) {
        int64_t gb, ge;
        group_range(gr, g, gb, ge);
        int64_t a = max(row, gb), b = min(r1, ge);
        float m = 0.0f;
        if (a < b) {
            const int64_t n = (b - a) * vec_per_row;
            for (int64_t i = threadIdx.x; i < n; i += kQuantThreads) {
                int64_t rr = a + i / vec_per_row;
                int v = (int)(i % vec_per_row);
                uint4 w = __ldg(reinterpret_cast<const uint4*>(x + rr * ldx) + v);
                m = fmaxf(m, fmaxf(fmaxf(fabsf(bf16lo(w.x)), fabsf(bf16hi(w.x))), fmaxf(fabsf(bf16lo(w.y)), fabsf(bf16hi(w.y)))));
                m = fmaxf(m, fmaxf(fmaxf(fabsf(bf16lo(w.z)), fabsf(bf16hi(w.z))), fmaxf(fabsf(bf16lo(w.w)), fabsf(bf16hi(w.w)))));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
        __syncthreads();
        if (threadIdx.x == 0) {
            float mm = 0.0f;
            for (int w = 0; w < kQuantThreads / 32; ++w) mm = fmaxf(mm, red[w]);
            if (a < b && mm > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(&ts[g].amax), __float_as_uint(mm));
        }
        __syncthreads();
        row = max(row, ge);
        ++g;
    }
}

// ------------------------------------------------------------------------ quantize + score
// BPT = 16-element blocks per thread along K (1 when K <= 4096, 2 when K <= 8192).
template <int BPT, bool kScores, int kWhat>  // kWhat: 0 none, 1 bf16 w_hat, 2 fp32 w_hat
__global__ void __launch_bounds__(kQuantThreads) quant_score_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t ldx, int K, Groups gr, int64_t rows_per_cta,
    uint8_t* __restrict__ codes, int64_t ld_codes, uint8_t* __restrict__ sf, int64_t sf_cols, int zero_pad,
    nvq_tensor_scale* __restrict__ ts, unsigned long long* __restrict__ scores, void* __restrict__ w_hat)
{
    extern __shared__ unsigned long long red_scores[];  // [kQuantThreads][16 * BPT] when needed
    const int nb = K / 16;
    const int lanes_per_row = (BPT == 1) ? nb : kQuantThreads;
    const int rows_per_iter = (BPT == 1) ? (kQuantThreads / nb) : 1;
    const int tid = threadIdx.x;
    const int rl = tid / lanes_per_row;
    const int bc0 = tid % lanes_per_row;
    const bool active = rl < rows_per_iter;

    // CTA 0 publishes every group's scale fields (amax is final: amax_kernel ran before).
    if (blockIdx.x == 0) {
        for (int g = tid; g < gr.G; g += kQuantThreads) {
            TScale t = tscale_from_amax(ts[g].amax);
            ts[g].s_enc = t.s_enc;
            ts[g].s_dec = t.s_dec;
            ts[g].shift_e = t.shift_e;
        }
    }

    const int64_t r0 = (int64_t)blockIdx.x * rows_per_cta;
    const int64_t r1 = min(r0 + rows_per_cta, gr.total_rows);
    if (r0 >= r1) return;
    int g = group_of_row(gr, r0);
    int64_t row = r0;
    while (row < r1 && g < gr.G) {
        int64_t gb, ge;
        group_range(gr, g, gb, ge);
        const int64_t a = max(row, gb), b = min(r1, ge);
        const TScale t = tscale_from_amax(ts[g].amax);
        const ScoreScale ss = score_scale(t.shift_e);
        unsigned long long part[BPT][16];
#pragma unroll
        for (int p = 0; p < BPT; ++p)
#pragma unroll
            for (int i = 0; i < 16; ++i) part[p][i] = 0ull;

        if (active) {
            for (int64_t r = a + rl; r < b; r += rows_per_iter) {
                const __nv_bfloat16* xr = x + r * ldx;
#pragma unroll
                for (int p = 0; p < BPT; ++p) {
                    const int bc = bc0 + p * kQuantThreads;
                    if (bc >= nb) continue;
                    const uint4* src = reinterpret_cast<const uint4*>(xr + bc * 16);
                    uint4 w0 = __ldg(src), w1 = __ldg(src + 1);
                    float v[16] = {bf16lo(w0.x), bf16hi(w0.x), bf16lo(w0.y), bf16hi(w0.y),
                                   bf16lo(w0.z), bf16hi(w0.z), bf16lo(w0.w), bf16hi(w0.w),
                                   bf16lo(w1.x), bf16hi(w1.x), bf16lo(w1.y), bf16hi(w1.y),
                                   bf16lo(w1.z), bf16hi(w1.z), bf16lo(w1.w), bf16hi(w1.w)};
                    BlockOut o = quantize16(v, t.s_enc, t.s_dec);
                    *reinterpret_cast<uint2*>(codes + r * ld_codes + bc * 8) = make_uint2(o.code_lo, o.code_hi);
                    sf[sf_offset(r, bc, sf_cols)] = (uint8_t)o.sb;
                    if (kScores || kWhat) {
                        float dq[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) dq[i] = __fmul_rn(e2m1_value(block_code(o, i)), o.d_b);
                        if (kScores) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) part[p][i] += score_term(__fsub_rn(v[i], dq[i]), ss);
                        }
                        if (kWhat == 1) {
                            uint32_t pk[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                __nv_bfloat162 h2 = __floats2bfloat162_rn(dq[2 * i], dq[2 * i + 1]);
                                pk[i] = *reinterpret_cast<uint32_t*>(&h2);
                            }
                            uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(w_hat) + r * (int64_t)K + bc * 16);
                            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                        } else if (kWhat == 2) {
                            float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(w_hat) + r * (int64_t)K + bc * 16);
#pragma unroll
                            for (int i = 0; i < 4; ++i) dst[i] = make_float4(dq[4 * i], dq[4 * i + 1], dq[4 * i + 2], dq[4 * i + 3]);
                        }
                    }
                }
                if (zero_pad && bc0 == 0) {
                    for (int64_t c = nb; c < sf_cols; ++c) sf[sf_offset(r, c, sf_cols)] = 0;
                }
            }
        }

        if (kScores) {
            unsigned long long* dst = scores + (int64_t)g * K;
            if (rows_per_iter == 1) {
                if (active && a < b) {
#pragma unroll
                    for (int p = 0; p < BPT; ++p) {
                        const int bc = bc0 + p * kQuantThreads;
                        if (bc >= nb) continue;
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (part[p][i]) atomicAdd(dst + bc * 16 + i, part[p][i]);
                    }
                }
            } else {
                // BPT == 1: fold the rows_per_iter row lanes of each block column in shared memory.
#pragma unroll
                for (int i = 0; i < 16; ++i) red_scores[tid * 16 + i] = part[0][i];
                __syncthreads();
                if (rl == 0 && a < b) {
#pragma unroll 1
                    for (int i = 0; i < 16; ++i) {
                        unsigned long long s = 0;
                        for (int l = 0; l < rows_per_iter; ++l) s += red_scores[(l * nb + bc0) * 16 + i];
                        if (s) atomicAdd(dst + bc0 * 16 + i, s);
                    }
                }
                __syncthreads();
            }
        }
        row = max(row, ge);
        ++g;
    }
}

// ------------------------------------------------------------------------ host side
struct QuantLaunch {
    int grid_amax, grid_quant;
    int64_t rpc_amax, rpc_quant;
};

static QuantLaunch plan(int64_t rows, int K)
{
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    QuantLaunch q;
    // amax: ~4 CTAs per SM, whole rows per CTA.
    int64_t want = (int64_t)sms * 4;
    q.rpc_amax = (rows + want - 1) / want;
    if (q.rpc_amax < 1) q.rpc_amax = 1;
    q.grid_amax = (int)((rows + q.rpc_amax - 1) / q.rpc_amax);
    // quantize: at least ~16 rows per CTA so that the score flush (K atomics per CTA) stays
    // small next to the data, and ~4 CTAs per SM.
    int64_t rpc = (rows + want - 1) / want;
    int64_t min_rows = (K >= 2048) ? 16 : 32;
    if (rpc < min_rows) rpc = min_rows;
    q.rpc_quant = rpc;
    q.grid_quant = (int)((rows + rpc - 1) / rpc);
    return q;
}

template <int BPT, bool S, int W>
static void launch_quant(const QuantLaunch& q, cudaStream_t st, const __nv_bfloat16* x, int64_t ldx, int K,
                         Groups gr, uint8_t* codes, int64_t ld_codes, uint8_t* sf, int64_t sf_cols,
                         int zero_pad, nvq_tensor_scale* ts, unsigned long long* scores, void* w_hat)
{
    size_t smem = (S && BPT == 1 && (kQuantThreads / (K / 16)) > 1) ? kQuantThreads * 16 * sizeof(unsigned long long) : 0;
    if (smem > 48 * 1024)
        cudaFuncSetAttribute(quant_score_kernel<BPT, S, W>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    quant_score_kernel<BPT, S, W><<<q.grid_quant, kQuantThreads, smem, st>>>(
        x, ldx, K, gr, q.rpc_quant, codes, ld_codes, sf, sf_cols, zero_pad, ts, scores, w_hat);
}

nvq_status quantize_impl(const void* x, int64_t rows, int64_t K, int64_t ldx, Groups gr, uint8_t* codes,
                         int64_t ld_codes, uint8_t* sf, int64_t sf_cols, int zero_pad, nvq_tensor_scale* ts,
                         uint64_t* scores, void* w_hat, int w_hat_dtype, cudaStream_t st)
{
    const QuantLaunch q = plan(rows, (int)K);
    cudaError_t e = cudaMemsetAsync(ts, 0, sizeof(nvq_tensor_scale) * gr.G, st);
    if (e != cudaSuccess) return cuda_status(e, "cudaMemsetAsync(tscale)");
    if (scores) {
        e = cudaMemsetAsync(scores, 0, sizeof(uint64_t) * gr.G * K, st);
        if (e != cudaSuccess) return cuda_status(e, "cudaMemsetAsync(scores)");
    }
    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
    amax_kernel<<<q.grid_amax, kQuantThreads, 0, st>>>(xb, ldx, (int)K, gr, q.rpc_amax, ts);
    NVQ_LAUNCH_CHECK("amax_kernel");
    unsigned long long* sc = reinterpret_cast<unsigned long long*>(scores);
    const int k = (int)K;
    const int what = w_hat ? (w_hat_dtype == NVQ_F32 ? 2 : 1) : 0;
    if (K <= 4096) {
        if (sc) launch_quant<1, true, 0>(q, st, xb, ldx, k, gr, codes, ld_codes, sf, sf_cols, zero_pad, ts, sc, nullptr);
        else if (what == 0) launch_quant<1, false, 0>(q, st, xb, ldx, k, gr, codes, ld_codes, sf, sf_cols, zero_pad, ts, nullptr, nullptr);
        else if (what == 1) launch_quant<1, false, 1>(q, st, xb, ldx, k, gr, codes, ld_codes, sf, sf_cols, zero_pad, ts, nullptr, w_hat);
        else launch_quant<1, false, 2>(q, st, xb, ldx, k, gr, codes, ld_codes, sf, sf_cols, zero_pad, ts, nullptr, w_hat);
    } else {
        if (sc) launch_quant<2, true, 0>(q, st, xb, ldx, k, gr, codes, ld_codes, sf, sf_cols, zero_pad, ts, sc, nullptr);
        else if (what == 0) launch_quant<2, false, 0>(q, st, xb, ldx, k, gr, codes, ld_codes, sf, sf_cols, zero_pad, ts, nullptr, nullptr);
        else if (what == 1) launch_quant<2, false, 1>(q, st, xb, ldx, k, gr, codes, ld_codes, sf, sf_cols, zero_pad, ts, nullptr, w_hat);
        else launch_quant<2, false, 2>(q, st, xb, ldx, k, gr, codes, ld_codes, sf, sf_cols, zero_pad, ts, nullptr, w_hat);
    }
    NVQ_LAUNCH_CHECK("quant_score_kernel");
    return NVQ_OK;
}

}  // namespace nvq

using namespace nvq;

extern "C" nvq_status nvfp4_quantize(const void* x, int64_t rows, int64_t K, int64_t ldx, const int64_t* grp_off,
                                     const int64_t* grp_rows, int32_t groups, uint8_t* codes, int64_t ld_codes,
                                     uint8_t* sf, int64_t sf_cols, int32_t zero_pad, nvq_tensor_scale* tscale,
                                     uint64_t* scores, void* stream)
{
    NVQ_CHECK_ARG(x && codes && sf && tscale, NVQ_ERR_ARG, "nvfp4_quantize: null pointer argument");
    NVQ_CHECK_ARG(rows >= 1 && rows <= (1ll << 24), NVQ_ERR_SHAPE, "nvfp4_quantize: rows=%lld outside [1, 2^24]", (long long)rows);
    NVQ_CHECK_ARG(K >= 16 && K <= 8192 && K % 16 == 0, NVQ_ERR_SHAPE, "nvfp4_quantize: K=%lld must be a multiple of 16 in [16, 8192]", (long long)K);
    NVQ_CHECK_ARG(groups >= 1 && groups <= 4096, NVQ_ERR_SHAPE, "nvfp4_quantize: groups=%d outside [1, 4096]", groups);
    NVQ_CHECK_ARG(grp_off || groups == 1 || rows % groups == 0, NVQ_ERR_SHAPE, "nvfp4_quantize: rows not divisible by groups");
    NVQ_CHECK_ARG(ldx >= K && ldx % 8 == 0, NVQ_ERR_ALIGN, "nvfp4_quantize: ldx=%lld must be >= K and a multiple of 8", (long long)ldx);
    NVQ_CHECK_ARG(ld_codes >= K / 2 && ld_codes % 16 == 0, NVQ_ERR_ALIGN, "nvfp4_quantize: ld_codes=%lld must be >= K/2 and a multiple of 16", (long long)ld_codes);
    NVQ_CHECK_ARG(sf_cols >= K / 16 && sf_cols % 4 == 0, NVQ_ERR_SHAPE, "nvfp4_quantize: sf_cols=%lld must be >= K/16 and a multiple of 4", (long long)sf_cols);
    NVQ_CHECK_ARG(aligned(x, 16) && aligned(codes, 16), NVQ_ERR_ALIGN, "nvfp4_quantize: x and codes must be 16-byte aligned");
    NVQ_CHECK_ARG(!scores || aligned(scores, 8), NVQ_ERR_ALIGN, "nvfp4_quantize: scores must be 8-byte aligned");
    Groups gr{grp_off, grp_rows, groups, rows};
    set_error("");
    return quantize_impl(x, rows, K, ldx, gr, codes, ld_codes, sf, sf_cols, zero_pad, tscale, scores, nullptr, 0,
                         static_cast<cudaStream_t>(stream));
}

extern "C" nvq_status weight_qdq(const void* w, int32_t groups, int64_t N, int64_t K, int64_t ldw, uint8_t* codes,
                                 int64_t ld_codes, uint8_t* sf, int64_t sf_cols, nvq_tensor_scale* tscale, void* w_hat,
                                 int32_t w_hat_dtype, void* stream)
{
    NVQ_CHECK_ARG(w && codes && sf && tscale, NVQ_ERR_ARG, "weight_qdq: null pointer argument");
    NVQ_CHECK_ARG(w_hat_dtype == NVQ_BF16 || w_hat_dtype == NVQ_F32, NVQ_ERR_ARG, "weight_qdq: w_hat_dtype must be NVQ_BF16 or NVQ_F32");
    NVQ_CHECK_ARG(groups >= 1 && groups <= 4096, NVQ_ERR_SHAPE, "weight_qdq: groups=%d outside [1, 4096]", groups);
    NVQ_CHECK_ARG(N >= 128 && N % 128 == 0, NVQ_ERR_SHAPE, "weight_qdq: N=%lld must be a positive multiple of 128", (long long)N);
    NVQ_CHECK_ARG((int64_t)groups * N <= (1ll << 24), NVQ_ERR_SHAPE, "weight_qdq: groups*N exceeds 2^24 rows");
    NVQ_CHECK_ARG(K >= 16 && K <= 8192 && K % 16 == 0, NVQ_ERR_SHAPE, "weight_qdq: K=%lld must be a multiple of 16 in [16, 8192]", (long long)K);
    NVQ_CHECK_ARG(ldw >= K && ldw % 8 == 0, NVQ_ERR_ALIGN, "weight_qdq: ldw must be >= K and a multiple of 8");
    NVQ_CHECK_ARG(ld_codes >= K / 2 && ld_codes % 16 == 0, NVQ_ERR_ALIGN, "weight_qdq: ld_codes must be >= K/2 and a multiple of 16");
    NVQ_CHECK_ARG(sf_cols >= K / 16 && sf_cols % 4 == 0, NVQ_ERR_SHAPE, "weight_qdq: sf_cols must be >= K/16 and a multiple of 4");
    NVQ_CHECK_ARG(aligned(w, 16) && aligned(codes, 16) && (!w_hat || aligned(w_hat, 16)), NVQ_ERR_ALIGN,
                  "weight_qdq: w, codes and w_hat must be 16-byte aligned");
    Groups gr{nullptr, nullptr, groups, (int64_t)groups * N};
    set_error("");
    return quantize_impl(w, (int64_t)groups * N, K, ldw, gr, codes, ld_codes, sf, sf_cols, 1, tscale, nullptr, w_hat,
                         w_hat_dtype, static_cast<cudaStream_t>(stream));
}
