// quantize.cu -- NVFP4 quantization of bf16 matrices (QUADS §2.2 "FP4"; Q_A of Eq. (9),
// Q_W of Eq. (7) and the trainer's QDQ_W of Eq. (12)) with the per-channel residual score of
// Eq. (23) fused into the same pass over the input.
//
// Two kernels per call (the first skipped when the producer of x measured the amax):
//   amax_kernel          per-group max |x| (the FP32 tensor scale's statistic), HBM-bound:
//                        16-byte loads marked evict-last in L2, 8 in flight per thread, one
//                        atomicMax per (CTA, group run);
//   quant_score_kernel   codes + blocked E4M3 scales + residual + integer channel score (+ the
//                        dequantized values for the trainer-side QDQ).  One CTA of 16 warps per
//                        SM: one lane streams the CTA's band of rows into a 5-stage shared
//                        memory ring of up to 32 KB stages with cp.async.bulk (up to 96 KB in
//                        flight per SM, independent of register pressure), every thread
//                        quantizes one 16-element block per row from shared memory, two or
//                        more rows per stage (fewer hand-offs per element).  The CTA re-reads the
//                        rows amax_kernel's CTAs just streamed, so most of that second read is
//                        served by L2.  Bound by instruction issue (the exact score costs about
//                        as much as the quantization), not by HBM.
#include <cuda_bf16.h>

#include "common.cuh"

namespace nvq {

// ------------------------------------------------------------------------ amax
static constexpr int kAmaxThreads = 256;
static constexpr int kAmaxUnroll = 8;

__device__ __forceinline__ float amax_u4(uint4 w)
{
    // |bf16| pairs as bf16x2 maxima (exact), then the two halves
    const uint32_t m = 0x7fff7fffu;
    __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162*>(&(w.x = w.x & m));
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&(w.y = w.y & m));
    __nv_bfloat162 c = *reinterpret_cast<__nv_bfloat162*>(&(w.z = w.z & m));
    __nv_bfloat162 d = *reinterpret_cast<__nv_bfloat162*>(&(w.w = w.w & m));
    __nv_bfloat162 r = __hmax2(__hmax2(a, b), __hmax2(c, d));
    return fmaxf(__low2float(r), __high2float(r));
}

// 16-byte load that marks its L2 lines evict-last: the quantize pass reads the same rows next,
// and an input up to about half of L2 then stays there for it.
__device__ __forceinline__ uint4 ld_keep(const uint4* p, uint64_t pol)
{
    uint4 v;
    asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}

__global__ void __launch_bounds__(kAmaxThreads) amax_kernel(const __nv_bfloat16* __restrict__ x, int64_t ldx, int K,
                                                             Groups gr, int64_t rows_per_cta,
                                                             nvq_tensor_scale* __restrict__ ts)
{
    __shared__ float red[kAmaxThreads / 32];
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    const int64_t r0 = (int64_t)blockIdx.x * rows_per_cta;
    const int64_t r1 = min(r0 + rows_per_cta, gr.total_rows);
    if (r0 >= r1) return;
    const int vpr = K / 8;  // 16-byte vectors per row
    int g = group_of_row(gr, r0);
    int64_t row = r0;
    while (row < r1 && g < gr.G) {
        int64_t gb, ge;
        group_range(gr, g, gb, ge);
        const int64_t a = max(row, gb), b = min(r1, ge);
        float m = 0.0f;
        if (a < b) {
            if (ldx == K) {
                // contiguous rows: one flat range of vectors
                const uint4* p = reinterpret_cast<const uint4*>(x + a * ldx);
                const int64_t n = (b - a) * vpr;
                int64_t i = threadIdx.x;
                for (; i + (kAmaxUnroll - 1) * kAmaxThreads < n; i += kAmaxUnroll * kAmaxThreads) {
                    uint4 w[kAmaxUnroll];
#pragma unroll
                    for (int u = 0; u < kAmaxUnroll; ++u) w[u] = ld_keep(p + i + u * kAmaxThreads, pol);
#pragma unroll
                    for (int u = 0; u < kAmaxUnroll; ++u) m = fmaxf(m, amax_u4(w[u]));
                }
                for (; i < n; i += kAmaxThreads) m = fmaxf(m, amax_u4(ld_keep(p + i, pol)));
            } else {
                for (int64_t r = a; r < b; ++r) {
                    const uint4* p = reinterpret_cast<const uint4*>(x + r * ldx);
                    for (int v = threadIdx.x; v < vpr; v += kAmaxThreads) m = fmaxf(m, amax_u4(ld_keep(p + v, pol)));
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
        __syncthreads();
        if (threadIdx.x == 0) {
            float mm = 0.0f;
            for (int w = 0; w < kAmaxThreads / 32; ++w) mm = fmaxf(mm, red[w]);
            if (a < b && mm > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(&ts[g].amax), __float_as_uint(mm));
        }
        __syncthreads();
        row = max(row, ge);
        ++g;
    }
}

// ------------------------------------------------------------------------ quantize + score
static constexpr int kQStages = 5;
static constexpr int kQStageBytes = 32768;  // capacity; a stage holds whole groups of rows_per_iter rows
static constexpr int kQCompute = 512;  // 16 warps: one thread per 16-element block up to K = 8192
static constexpr int kQThreads = kQCompute;
static constexpr int kQAhead = kQStages - 2;  // stages the loads run ahead of the compute
static constexpr int kQLoader = kQThreads - 32;  // the thread that issues the bulk copies (warp 15, lane 0)

__device__ __forceinline__ uint32_t sa32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void q_mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa32(bar)), "r"(count));
}

__device__ __forceinline__ bool q_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(sa32(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// Non-blocking test of the phase (try_wait may suspend the thread in hardware for a while).
__device__ __forceinline__ bool q_test_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(sa32(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}

// A bound shorter than this polls with test_wait, so that it is honoured to within a poll
// instead of the hardware's suspend window of try_wait.
constexpr unsigned long long kShortWaitCycles = 1ull << 20;

// Bounded wait: false after recording a timeout, or (unless draining) as soon as another warp
// of the CTA gave up.
__device__ __forceinline__ bool q_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, DeviceStatus* st,
                                       unsigned long long limit, int where, bool draining = false)
{
    const unsigned long long bound = draining ? drain_limit(limit) : limit;
    const bool poll = bound < kShortWaitCycles;
    if (poll ? q_test_wait(bar, parity) : q_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        // the bound is checked before each round of polls, so that a limit of a few cycles
        // runs out at the first wait that is not already complete
        if (!draining && *abort_flag) return false;
        if ((unsigned long long)(clock64() - t0) > bound) {
            report_timeout(st, where);
            *abort_flag = 1;
            return false;
        }
        for (int i = 0; i < 32; ++i)
            if (poll ? q_test_wait(bar, parity) : q_try_wait(bar, parity)) return true;
    }
}

// Bulk copy of rows into the ring with a cache policy: normal priority (the lines the amax
// pass marked evict-last go back to normal once consumed), or evict-last when the amax came
// from the producer and the residual tail will read the rows again.
__device__ __forceinline__ void q_bulk_row(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
                     sa32(dst)),
                 "l"(src), "r"(bytes), "r"(sa32(bar)), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kQCompute) : "memory"); }

// fl(a / 6) for a non-negative bf16 value a, without a division: the quotient estimate
// q1 = fl(a * fl(1/6)) is corrected once with fused multiply-adds, as in Markstein's
// FMA-based division (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Develop. 34(1), 1990): the remainder r = a - 6 q1 is exact
// in one FMA, and q1 + r * fl(1/6) rounds to the correctly rounded quotient.  That this holds
// for every finite non-negative bf16 input is checked exhaustively against the IEEE division
// __fdiv_rn by nvq_check_block_scale_division.
__device__ __forceinline__ float div6_bf16(float a)
{
    constexpr float kInv6 = 1.0f / 6.0f;
    const float q1 = __fmul_rn(a, kInv6);
    const float r = __fmaf_rn(-q1, 6.0f, a);
    return __fmaf_rn(r, kInv6, q1);
}

// max(|a|, |b|) of two bf16x2 words per half (exact; the sign bits of the result are the
// XOR of the inputs' and are cleared by the caller).
__device__ __forceinline__ uint32_t max_abs_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Block amax of 16 bf16 values held as 8 bf16x2 words, as an fp32 value (exact).
__device__ __forceinline__ float block_amax_words(const uint32_t* w)
{
    const uint32_t m = max_abs_bf16x2(max_abs_bf16x2(max_abs_bf16x2(w[0], w[1]), max_abs_bf16x2(w[2], w[3])),
                                      max_abs_bf16x2(max_abs_bf16x2(w[4], w[5]), max_abs_bf16x2(w[6], w[7]))) &
                       0x7fff7fffu;
    return fmaxf(bf16lo(m), bf16hi(m));
}

// Eight fp32 values (four pairs, element 2i in the low word of pair i) -> eight E2M1 codes in
// one word, element 2i in the low nibble of byte i (round to nearest even, saturate, sign kept).
__device__ __forceinline__ uint32_t e2m1x8(const uint64_t* yp)
{
    float y[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) f2unpack(yp[i], y[2 * i], y[2 * i + 1]);
    uint32_t w;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(w)
        : "f"(y[0]), "f"(y[1]), "f"(y[2]), "f"(y[3]), "f"(y[4]), "f"(y[5]), "f"(y[6]), "f"(y[7]));
    return w;
}

// Byte j of a code word -> the two E2M1 values as an fp32 pair (exact).
__device__ __forceinline__ uint64_t e2m1_byte_to_f2(uint32_t w, int j)
{
    uint32_t h;
    switch (j) {
    case 0: asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b0;\n\t}" : "=r"(h) : "r"(w)); break;
    case 1: asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b1;\n\t}" : "=r"(h) : "r"(w)); break;
    case 2: asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b2;\n\t}" : "=r"(h) : "r"(w)); break;
    default: asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b3;\n\t}" : "=r"(h) : "r"(w)); break;
    }
    const float2 v = __half22float2(*reinterpret_cast<__half2*>(&h));
    return f2pack(v.x, v.y);
}

// acc += q^2 for a signed q with |q| < 2^19: one 32 x 32 -> 64-bit multiply-add.
__device__ __forceinline__ void score_acc_signed(unsigned long long& acc, int q)
{
    asm("mad.wide.s32 %0, %1, %1, %0;" : "+l"(acc) : "r"(q));
}

struct QuantArgs {
    const __nv_bfloat16* x;
    int64_t ldx;
    int K;
    Groups gr;
    int64_t rows_per_cta;
    uint8_t* codes;
    int64_t ld_codes;
    uint8_t* sf;
    int64_t sf_cols;
    int zero_pad;
    nvq_tensor_scale* ts;
    unsigned long long* scores;
    void* w_hat;
    DeviceStatus* status;
    unsigned long long wait_limit;
    int keep_l2;  // mark the rows evict-last (the residual tail re-reads them) instead of normal
};

// BPT = 16-element blocks per thread along K (1: K / 16 <= kQCompute).
// Producer cursor: walks the CTA's band of rows in the same order as the compute loop (group run
// by group run, R rows per stage) and issues each stage's bulk copies.
struct LoadCursor {
    int g;
    int64_t row, r, b;  // current group run [r, b) of the band, next stage starts at r
    uint32_t it;        // stages issued so far
    bool done;
};

__device__ __forceinline__ void cursor_next_run(const QuantArgs& qa, LoadCursor& c, int64_t r1)
{
    // advance to the first non-empty group run at or after c.row
    while (c.row < r1 && c.g < qa.gr.G) {
        int64_t gb, ge;
        group_range(qa.gr, c.g, gb, ge);
        const int64_t a = max(c.row, gb), b = min(r1, ge);
        if (a < b) {
            c.r = a;
            c.b = b;
            return;
        }
        c.row = max(c.row, ge);
        ++c.g;
    }
    c.done = true;
}

// Issue the loads of stage c.it if the compute has released its ring slot (bounded wait).
__device__ __forceinline__ bool cursor_issue(const QuantArgs& qa, LoadCursor& c, int64_t r1, int R, int row_bytes,
                                             uint8_t* ring, uint64_t* full_bar, uint64_t* empty_bar, volatile int* abrt)
{
    const int s = c.it % kQStages;
    if (c.it >= kQStages &&
        !q_wait(&empty_bar[s], ((c.it / kQStages) & 1) ^ 1, abrt, qa.status, qa.wait_limit, 21))
        return false;
    const int nr = (int)min((int64_t)R, c.b - c.r);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(sa32(&full_bar[s])),
                 "r"((uint32_t)(nr * row_bytes))
                 : "memory");
    uint64_t pol;
    if (qa.keep_l2)
        asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    else
        asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    if (qa.ldx * 2 == row_bytes)  // contiguous rows: the whole stage in one copy
        q_bulk_row(ring + s * kQStageBytes, qa.x + c.r * qa.ldx, (uint32_t)(nr * row_bytes), &full_bar[s], pol);
    else
        for (int j = 0; j < nr; ++j)
            q_bulk_row(ring + s * kQStageBytes + j * row_bytes, qa.x + (c.r + j) * qa.ldx, row_bytes, &full_bar[s], pol);
    ++c.it;
    c.r += R;
    if (c.r >= c.b) {
        c.row = c.b;
        int64_t gb, ge;
        group_range(qa.gr, c.g, gb, ge);
        c.row = max(c.row, ge);
        ++c.g;
        cursor_next_run(qa, c, r1);
    }
    return true;
}

// One CTA of 16 warps per SM (4 per scheduler, 128 registers a thread: the 16 exact 64-bit
// channel-score accumulators a thread holds stay in registers).  Every warp computes; lane 0 of
// warp 15 also issues the bulk copies kQAhead stages ahead of the compute.
template <int BPT, bool kScores, int kWhat>  // kWhat: 0 none, 1 bf16 w_hat, 2 fp32 w_hat
__global__ void __launch_bounds__(kQThreads, 1) quant_score_kernel(const QuantArgs qa)
{
    extern __shared__ __align__(128) uint8_t ring[];
    __shared__ __align__(8) uint64_t full_bar[kQStages], empty_bar[kQStages];
    __shared__ float eb_tab[128], db_tab[128];
    __shared__ int abort_flag;

    const int K = qa.K;
    const int nb = K / 16;
    const int row_bytes = 2 * K;
    // rows per stage: whole groups of the rows_per_iter rows the threads take side by side, as
    // many as fit, so every thread handles the same number of rows per stage
    const int rpi = (BPT == 1) ? (kQCompute / nb) : 1;
    const int R = rpi * max(1, kQStageBytes / (rpi * row_bytes));
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    unsigned long long* red_scores = reinterpret_cast<unsigned long long*>(ring + kQStages * kQStageBytes);

    if (tid == 0) {
        for (int i = 0; i < kQStages; ++i) {
            q_mbar_init(&full_bar[i], 1);
            q_mbar_init(&empty_bar[i], kQCompute / 32);
        }
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // CTA 0 publishes every group's scale fields (amax is final: amax_kernel ran before).
    if (blockIdx.x == 0) {
        for (int g = tid; g < qa.gr.G; g += kQThreads) {
            TScale t = tscale_from_amax(qa.ts[g].amax);
            qa.ts[g].s_enc = t.s_enc;
            qa.ts[g].s_dec = t.s_dec;
            qa.ts[g].shift_e = t.shift_e;
        }
    }
    __syncthreads();
    volatile int* abrt = &abort_flag;

    const int64_t r0 = (int64_t)blockIdx.x * qa.rows_per_cta;
    const int64_t r1 = min(r0 + qa.rows_per_cta, qa.gr.total_rows);
    if (r0 >= r1) return;

    // ---------------- loader prologue: the first kQAhead stages
    const bool loader = tid == kQLoader;
    LoadCursor cur;
    cur.g = group_of_row(qa.gr, r0);
    cur.row = r0;
    cur.r = cur.b = 0;
    cur.it = 0;
    cur.done = false;
    bool load_ok = true;
    if (loader) {
        cursor_next_run(qa, cur, r1);
        while (load_ok && !cur.done && cur.it < (uint32_t)kQAhead)
            load_ok = cursor_issue(qa, cur, r1, R, row_bytes, ring, full_bar, empty_bar, abrt);
    }

    // ---------------- compute (all warps)
    const int lanes_per_row = (BPT == 1) ? nb : kQCompute;
    const int rows_per_iter = (BPT == 1) ? (kQCompute / nb) : 1;
    const int rl = tid / lanes_per_row;
    const int bc0 = tid % lanes_per_row;
    const bool active = rl < rows_per_iter;
    bool dead = false;
    uint32_t it = 0;
    int g = group_of_row(qa.gr, r0);
    int64_t row = r0;
    while (row < r1 && g < qa.gr.G) {
        int64_t gb, ge;
        group_range(qa.gr, g, gb, ge);
        const int64_t a = max(row, gb), b = min(r1, ge);
        const TScale t = tscale_from_amax(qa.ts[g].amax);
        const ScoreScale ss = score_scale(t.shift_e);
        // per-group encode / decode scale of every E4M3 block-scale value
        consumer_sync();
        if (tid < 128) {
            const float sbv = e4m3_value((uint32_t)tid);
            eb_tab[tid] = (tid == 0 || tid == 127) ? 0.0f : encode_factor(t.s_enc, sbv);
            db_tab[tid] = (tid == 127) ? 0.0f : __fmul_rn(sbv, t.s_dec);
        }
        consumer_sync();
        unsigned long long part[BPT][16];
#pragma unroll
        for (int p = 0; p < BPT; ++p)
#pragma unroll
            for (int i = 0; i < 16; ++i) part[p][i] = 0ull;

        for (int64_t r = a; r < b; r += R, ++it) {
            const int s = it % kQStages;
            // keep the loads kQAhead stages ahead (the slot refilled here was released two stages ago)
            if (loader && load_ok && !cur.done && !*abrt)
                load_ok = cursor_issue(qa, cur, r1, R, row_bytes, ring, full_bar, empty_bar, abrt);
            // a warp that gives up keeps walking the same sequence (so that no named barrier is
            // left waiting for it) but skips the work
            if (!dead && !q_wait(&full_bar[s], (it / kQStages) & 1, abrt, qa.status, qa.wait_limit, 23)) dead = true;
            const int nr = (int)min((int64_t)R, b - r);
            const uint8_t* stage = ring + s * kQStageBytes;
            if (active && !dead) {
                for (int rr = rl; rr < nr; rr += rows_per_iter) {
                    const int64_t grow = r + rr;
                    uint8_t* crow = qa.codes + grow * qa.ld_codes;
                    const int64_t sfrow = (grow >> 7) * (qa.sf_cols >> 2) * 512 + (grow & 31) * 16 + ((grow >> 5) & 3) * 4;
#pragma unroll
                    for (int p = 0; p < BPT; ++p) {
                        const int bc = bc0 + p * kQCompute;
                        if (bc >= nb) continue;
                        const uint4* src = reinterpret_cast<const uint4*>(stage + rr * row_bytes + bc * 32);
                        const uint4 w0 = src[0], w1 = src[1];
                        const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
                        const uint32_t sb = e4m3(__fmul_rn(div6_bf16(block_amax_words(wv)), t.s_enc));
                        // sb == 0: e_b = 0 turns every x into a signed zero (code 0x0 / 0x8) and
                        // d_b = 0 makes the dequantized value 0, so no branch is needed
                        const float e_b = eb_tab[sb], d_b = db_tab[sb];
                        const uint64_t e2 = f2pack(e_b, e_b);
                        uint64_t xp[8], yp[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            xp[i] = bf16x2_to_f2(wv[i]);
                            yp[i] = f2mul(xp[i], e2);
                        }
                        const uint32_t lo = e2m1x8(yp), hi = e2m1x8(yp + 4);
                        *reinterpret_cast<uint2*>(crow + bc * 8) = make_uint2(lo, hi);
                        qa.sf[sfrow + (bc >> 2) * 512 + (bc & 3)] = (uint8_t)sb;
                        if (kScores || kWhat) {
                            const uint64_t d2 = f2pack(d_b, d_b);
                            uint64_t dq[8];  // fl(V[q] * d_b), pairs
#pragma unroll
                            for (int i = 0; i < 8; ++i) dq[i] = f2mul(e2m1_byte_to_f2(i < 4 ? lo : hi, i & 3), d2);
                            if (kScores) {
                                if (!ss.split) {
                                    // rint(r * sc) by the magic-number addition: 1.5 * 2^23 is even, so
                                    // the sum rounds to 1.5 * 2^23 + rint(r * sc) (ties to even) and its
                                    // bit pattern minus that of 1.5 * 2^23 is the signed integer, whose
                                    // square is rint(|r| * sc)^2
                                    const uint64_t sc2 = f2pack(ss.sc_a, ss.sc_a);
                                    const uint64_t m2 = f2pack(12582912.0f, 12582912.0f);
#pragma unroll
                                    for (int i = 0; i < 8; ++i) {
                                        float t0, t1;
                                        f2unpack(f2fma(f2sub(xp[i], dq[i]), sc2, m2), t0, t1);
                                        score_acc_signed(part[p][2 * i], __float_as_int(t0) - 0x4B400000);
                                        score_acc_signed(part[p][2 * i + 1], __float_as_int(t1) - 0x4B400000);
                                    }
                                } else {
#pragma unroll
                                    for (int i = 0; i < 8; ++i) {
                                        float x0, x1, q0, q1;
                                        f2unpack(xp[i], x0, x1);
                                        f2unpack(dq[i], q0, q1);
                                        part[p][2 * i] += score_term(__fsub_rn(x0, q0), ss);
                                        part[p][2 * i + 1] += score_term(__fsub_rn(x1, q1), ss);
                                    }
                                }
                            }
                            if (kWhat == 1) {
                                uint32_t pk[8];
#pragma unroll
                                for (int i = 0; i < 8; ++i) {
                                    float q0, q1;
                                    f2unpack(dq[i], q0, q1);
                                    __nv_bfloat162 h2 = __floats2bfloat162_rn(q0, q1);
                                    pk[i] = *reinterpret_cast<uint32_t*>(&h2);
                                }
                                uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(qa.w_hat) + grow * (int64_t)K + bc * 16);
                                dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                                dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                            } else if (kWhat == 2) {
                                float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(qa.w_hat) + grow * (int64_t)K + bc * 16);
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    float a0, a1, b0, b1;
                                    f2unpack(dq[2 * i], a0, a1);
                                    f2unpack(dq[2 * i + 1], b0, b1);
                                    dst[i] = make_float4(a0, a1, b0, b1);
                                }
                            }
                        }
                    }
                    if (qa.zero_pad && bc0 == 0)
                        for (int64_t cc = nb; cc < qa.sf_cols; ++cc) qa.sf[sf_offset(grow, cc, qa.sf_cols)] = 0;
                }
            }
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(sa32(&empty_bar[s])) : "memory");
        }

        if (kScores) {
            unsigned long long* dst = qa.scores + (int64_t)g * K;
            if (rows_per_iter == 1) {
                if (active && a < b && !dead) {
#pragma unroll
                    for (int p = 0; p < BPT; ++p) {
                        const int bc = bc0 + p * kQCompute;
                        if (bc >= nb) continue;
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (part[p][i]) atomicAdd(dst + bc * 16 + i, part[p][i]);
                    }
                }
            } else {
                // BPT == 1: fold the rows_per_iter row lanes of each channel in shared memory,
                // one channel per compute thread at a time
#pragma unroll
                for (int i = 0; i < 16; ++i) red_scores[tid * 16 + i] = part[0][i];
                consumer_sync();
                if (a < b && !dead) {
                    for (int ch = tid; ch < K; ch += kQCompute) {
                        unsigned long long sum = 0;
                        for (int l = 0; l < rows_per_iter; ++l) sum += red_scores[l * K + ch];
                        if (sum) atomicAdd(dst + ch, sum);
                    }
                }
                consumer_sync();
            }
        }
        row = max(row, ge);
        ++g;
    }
    if (loader && *abrt) {
        // after a timeout, let the copies still in flight land before the CTA exits (the last
        // issue on each slot)
        for (uint32_t j = cur.it > kQStages ? cur.it - kQStages : 0; j < cur.it; ++j)
            q_wait(&full_bar[j % kQStages], (j / kQStages) & 1, abrt, qa.status, qa.wait_limit, 22, true);
    }
}

// ------------------------------------------------------------------------ self-check
// Every finite non-negative bf16 bit pattern (0x0000 .. 0x7f7f) through div6_bf16 and through
// the IEEE division; out[0] counts the inputs whose results differ, out[1] keeps the lowest such
// pattern (0xffffffff when there is none).
__global__ void __launch_bounds__(256) div6_check_kernel(unsigned int* __restrict__ out)
{
    const uint32_t b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b > 0x7f7fu) return;
    const float a = __uint_as_float(b << 16);
    if (__float_as_uint(div6_bf16(a)) != __float_as_uint(__fdiv_rn(a, 6.0f))) {
        atomicAdd(&out[0], 1u);
        atomicMin(&out[1], b);
    }
}

// ------------------------------------------------------------------------ host side
static int sm_count()
{
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

template <int BPT, bool S, int W>
static cudaError_t launch_quant(int grid, cudaStream_t st, const QuantArgs& qa)
{
    const size_t smem = (size_t)kQStages * kQStageBytes + (S ? kQCompute * 16 * sizeof(unsigned long long) : 0);
    cudaError_t e = cudaFuncSetAttribute(quant_score_kernel<BPT, S, W>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    quant_score_kernel<BPT, S, W><<<grid, kQThreads, smem, st>>>(qa);
    return cudaGetLastError();
}

// amax: ~8 CTAs per SM, whole rows per CTA, atomically folded into ts[g].amax (zeroed before).
static nvq_status launch_amax(const __nv_bfloat16* x, int64_t rows, int64_t K, int64_t ldx, Groups gr,
                              nvq_tensor_scale* ts, int sms, cudaStream_t st)
{
    const int64_t want = (int64_t)sms * 8;
    int64_t rpc = (rows + want - 1) / want;
    if (rpc < 1) rpc = 1;
    const int grid = (int)((rows + rpc - 1) / rpc);
    amax_kernel<<<grid, kAmaxThreads, 0, st>>>(x, ldx, (int)K, gr, rpc, ts);
    NVQ_LAUNCH_CHECK("amax_kernel");
    return NVQ_OK;
}

nvq_status quantize_impl(const void* x, int64_t rows, int64_t K, int64_t ldx, Groups gr, uint8_t* codes,
                         int64_t ld_codes, uint8_t* sf, int64_t sf_cols, int zero_pad, nvq_tensor_scale* ts,
                         uint64_t* scores, void* w_hat, int w_hat_dtype, cudaStream_t st, bool amax_given = false)
{
    const int sms = sm_count();
    cudaError_t e = cudaSuccess;
    if (!amax_given) {
        e = cudaMemsetAsync(ts, 0, sizeof(nvq_tensor_scale) * gr.G, st);
        if (e != cudaSuccess) return cuda_status(e, "cudaMemsetAsync(tscale)");
    }
    if (scores) {
        e = cudaMemsetAsync(scores, 0, sizeof(uint64_t) * gr.G * K, st);
        if (e != cudaSuccess) return cuda_status(e, "cudaMemsetAsync(scores)");
    }
    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
    // amax (skipped when the producer of x computed it)
    if (!amax_given) {
        const nvq_status s = launch_amax(xb, rows, K, ldx, gr, ts, sms, st);
        if (s != NVQ_OK) return s;
    }
    QuantArgs qa;
    qa.x = xb;
    qa.ldx = ldx;
    qa.K = (int)K;
    qa.gr = gr;
    qa.rows_per_cta = (rows + sms - 1) / sms;
    qa.codes = codes;
    qa.ld_codes = ld_codes;
    qa.sf = sf;
    qa.sf_cols = sf_cols;
    qa.zero_pad = zero_pad;
    qa.ts = ts;
    qa.scores = reinterpret_cast<unsigned long long*>(scores);
    qa.w_hat = w_hat;
    qa.status = device_status_ptr();
    qa.wait_limit = wait_limit();
    // with the amax given there was no amax pass to leave x in L2: keep what fits for the
    // residual tail, which reads part of every row again (and demotes the lines as it goes)
    qa.keep_l2 = (amax_given && scores) ? 1 : 0;
    NVQ_CHECK_ARG(qa.status, NVQ_ERR_CUDA, "quantize: device status word unavailable");
    const int grid = (int)((rows + qa.rows_per_cta - 1) / qa.rows_per_cta);
    const bool sc = scores != nullptr;
    const int what = w_hat ? (w_hat_dtype == NVQ_F32 ? 2 : 1) : 0;
    static_assert(kQCompute * 16 >= 8192, "one 16-element block per thread must cover K <= 8192");
    if (sc) e = launch_quant<1, true, 0>(grid, st, qa);
    else if (what == 0) e = launch_quant<1, false, 0>(grid, st, qa);
    else if (what == 1) e = launch_quant<1, false, 1>(grid, st, qa);
    else e = launch_quant<1, false, 2>(grid, st, qa);
    if (e != cudaSuccess) return cuda_status(e, "quant_score_kernel");
    return NVQ_OK;
}

}  // namespace nvq

using namespace nvq;

extern "C" nvq_status nvfp4_quantize(const void* x, int64_t rows, int64_t K, int64_t ldx, const int64_t* grp_off,
                                     const int64_t* grp_rows, int32_t groups, uint8_t* codes, int64_t ld_codes,
                                     uint8_t* sf, int64_t sf_cols, int32_t zero_pad, nvq_tensor_scale* tscale,
                                     uint64_t* scores, int32_t amax_given, void* stream)
{
    NVQ_TRACE("nvfp4_quantize");
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
                         static_cast<cudaStream_t>(stream), amax_given != 0);
}

extern "C" nvq_status weight_qdq(const void* w, int32_t groups, int64_t N, int64_t K, int64_t ldw, uint8_t* codes,
                                 int64_t ld_codes, uint8_t* sf, int64_t sf_cols, nvq_tensor_scale* tscale, void* w_hat,
                                 int32_t w_hat_dtype, void* stream)
{
    NVQ_TRACE("weight_qdq");
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

extern "C" nvq_status nvfp4_amax(const void* x, int64_t rows, int64_t K, int64_t ldx, const int64_t* grp_off,
                                 const int64_t* grp_rows, int32_t groups, nvq_tensor_scale* tscale, void* stream)
{
    NVQ_TRACE("nvfp4_amax");
    NVQ_CHECK_ARG(x && tscale, NVQ_ERR_ARG, "nvfp4_amax: null pointer argument");
    NVQ_CHECK_ARG(rows >= 1 && rows <= (1ll << 24), NVQ_ERR_SHAPE, "nvfp4_amax: rows=%lld outside [1, 2^24]", (long long)rows);
    NVQ_CHECK_ARG(K >= 16 && K <= 8192 && K % 16 == 0, NVQ_ERR_SHAPE, "nvfp4_amax: K=%lld must be a multiple of 16 in [16, 8192]", (long long)K);
    NVQ_CHECK_ARG(groups >= 1 && groups <= 4096, NVQ_ERR_SHAPE, "nvfp4_amax: groups=%d outside [1, 4096]", groups);
    NVQ_CHECK_ARG(grp_off || groups == 1 || rows % groups == 0, NVQ_ERR_SHAPE, "nvfp4_amax: rows not divisible by groups");
    NVQ_CHECK_ARG(ldx >= K && ldx % 8 == 0, NVQ_ERR_ALIGN, "nvfp4_amax: ldx=%lld must be >= K and a multiple of 8", (long long)ldx);
    NVQ_CHECK_ARG(aligned(x, 16), NVQ_ERR_ALIGN, "nvfp4_amax: x must be 16-byte aligned");
    set_error("");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const cudaError_t e = cudaMemsetAsync(tscale, 0, sizeof(nvq_tensor_scale) * groups, st);
    if (e != cudaSuccess) return cuda_status(e, "cudaMemsetAsync(tscale)");
    return launch_amax(static_cast<const __nv_bfloat16*>(x), rows, K, ldx, Groups{grp_off, grp_rows, groups, rows}, tscale,
                       sm_count(), st);
}

extern "C" nvq_status nvq_check_block_scale_division(uint32_t* result, void* stream)
{
    NVQ_TRACE("nvq_check_block_scale_division");
    NVQ_CHECK_ARG(result, NVQ_ERR_ARG, "nvq_check_block_scale_division: null result pointer");
    NVQ_CHECK_ARG(aligned(result, 4), NVQ_ERR_ALIGN, "nvq_check_block_scale_division: result must be 4-byte aligned");
    set_error("");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(result, 0, sizeof(uint32_t), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(result + 1, 0xff, sizeof(uint32_t), st);
    if (e != cudaSuccess) return cuda_status(e, "cudaMemsetAsync(result)");
    div6_check_kernel<<<(0x7f80 + 255) / 256, 256, 0, st>>>(reinterpret_cast<unsigned int*>(result));
    NVQ_LAUNCH_CHECK("div6_check_kernel");
    return NVQ_OK;
}
