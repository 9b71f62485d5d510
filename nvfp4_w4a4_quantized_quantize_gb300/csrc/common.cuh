// common.cuh -- device helpers shared by the library's kernels (sm_103a).
//
// NVFP4 as in QUADS (arXiv 2607.15810) §2.2 "FP4": E2M1 element codes, one E4M3 block scale
// per 16 elements along K, one FP32 tensor scale.  The quantizer's operation order is:
//   S_enc = fl(2688 / amax), S_dec = fl(1 / S_enc)            (amax 0 -> 1, 1)
//   sb    = e4m3_rn_satfinite(fl(fl(amax_b / 6) * S_enc))
//   q     = e2m1_rn_satfinite(fl(x * fl(S_enc / sb)))          (sb == 0 -> +-0)
//   DQ(q) = fl(V[q] * fl(sb * S_dec)),  r = fl(x - DQ(q))
// Every step is written with explicit round-to-nearest intrinsics so that nvcc cannot contract
// a multiply and an add into an FMA.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stdint.h>

#include "../../include/nvfp4rac.h"

namespace nvq {

// ------------------------------------------------------------------ host-side error plumbing
void set_error(const char* fmt, ...);
nvq_status cuda_status(cudaError_t e, const char* what);
// Device status word (NVQ_OK / NVQ_ERR_TIMEOUT) and the wait bound in clock cycles.
struct DeviceStatus {
    int32_t status;
    int32_t where;
};
DeviceStatus* device_status_ptr();   // address of the current device's status word
unsigned long long wait_limit();      // cycles
int tail_path();                      // nvq_tail_path set by nvq_set_tail_path

#define NVQ_CHECK_ARG(cond, code, ...)          \
    do {                                        \
        if (!(cond)) {                          \
            ::nvq::set_error(__VA_ARGS__);      \
            return code;                        \
        }                                       \
    } while (0)

// NVTX range around one API call, named after the entry point: Nsight Systems and Nsight
// Compute (--nvtx) show each call's kernels under it.  With no tool attached a push or pop is a
// test of one function pointer.
struct TraceRange {
    explicit TraceRange(const char* name) { nvtxRangePushA(name); }
    ~TraceRange() { nvtxRangePop(); }
    TraceRange(const TraceRange&) = delete;
    TraceRange& operator=(const TraceRange&) = delete;
};
#define NVQ_TRACE(name) ::nvq::TraceRange nvq_trace_range_(name)

#define NVQ_LAUNCH_CHECK(what)                                             \
    do {                                                                   \
        cudaError_t e_ = cudaGetLastError();                               \
        if (e_ != cudaSuccess) return ::nvq::cuda_status(e_, what);        \
    } while (0)

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ------------------------------------------------------------------ blocked scale layout
__host__ __device__ __forceinline__ int64_t sf_offset(int64_t r, int64_t c, int64_t sf_cols)
{
    return ((r >> 7) * (sf_cols >> 2) + (c >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (c & 3);
}

// ------------------------------------------------------------------ row groups
struct Groups {
    const int64_t* off;   // [G+1] or nullptr
    const int64_t* rows;  // [G] or nullptr
    int32_t G;
    int64_t total_rows;   // rows extent of the matrix
};

// Row range [begin, end) of group g.
__device__ __forceinline__ void group_range(const Groups& gr, int g, int64_t& begin, int64_t& end)
{
    if (gr.off == nullptr) {
        int64_t per = gr.total_rows / gr.G;
        begin = per * g;
        end = begin + per;
    } else {
        begin = gr.off[g];
        end = gr.rows ? begin + gr.rows[g] : gr.off[g + 1];
    }
}

// Last group whose start is <= row (groups are sorted by start).
__device__ __forceinline__ int group_of_row(const Groups& gr, int64_t row)
{
    if (gr.G == 1) return 0;
    if (gr.off == nullptr) {
        int64_t per = gr.total_rows / gr.G;
        int g = (int)(row / per);
        return g < gr.G ? g : gr.G - 1;
    }
    int lo = 0, hi = gr.G - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (gr.off[mid] <= row) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// ------------------------------------------------------------------ tensor scale
struct TScale {
    float s_enc, s_dec;
    int32_t shift_e;
};

__device__ __forceinline__ TScale tscale_from_amax(float amax)
{
    TScale t;
    if (amax == 0.0f) {
        t.s_enc = 1.0f;
        t.s_dec = 1.0f;
        t.shift_e = 0;
    } else {
        float s = __fdiv_rn(2688.0f, amax);
        if (isinf(s)) s = 3.4028234663852886e38f;
        t.s_enc = s;
        t.s_dec = __fdiv_rn(1.0f, s);
        t.shift_e = ilogbf(amax) + 2;
    }
    return t;
}

// ------------------------------------------------------------------ element conversions
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two fp32 -> two E2M1 codes in one byte (lo -> low nibble), round to nearest even, saturate.
// The conversion keeps the sign of inputs that round to zero (-0 and small negatives give
// 0x8), which is the sign convention of the codes; the GB300 tests check every bf16 input.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi)
{
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

// fp32 (>= 0) -> E4M3 byte, round to nearest even, saturating at 448.
__device__ __forceinline__ uint32_t e4m3(float t)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(t));
    return (uint32_t)r & 0xffu;
}

// E4M3 byte -> fp32 (exact).
__device__ __forceinline__ float e4m3_value(uint32_t b)
{
    uint32_t h;
    uint16_t in = (uint16_t)(b & 0xffu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(in));
    return __half2float(__ushort_as_half((unsigned short)(h & 0xffffu)));
}

// One E2M1 code -> fp32 magnitude-with-sign (exact), via a two-word byte table.
__device__ __forceinline__ float e2m1_value(uint32_t c)
{
    // bf16 high halves of {0, .5, 1, 1.5, 2, 3, 4, 6}: 0000 3f00 3f80 3fc0 4000 4040 4080 40c0
    const uint32_t hi_lo = 0x3f3f3f00u, hi_hi = 0x40404040u;  // byte 1 of each bf16
    const uint32_t lo_lo = 0xc0800000u, lo_hi = 0xc0804000u;  // byte 0 of each bf16
    uint32_t m = c & 7u;
    uint32_t hb = __byte_perm(hi_lo, hi_hi, m);
    uint32_t lb = __byte_perm(lo_lo, lo_hi, m);
    uint32_t bits = ((hb & 0xffu) << 24) | ((lb & 0xffu) << 16) | ((c & 8u) << 28);
    return __uint_as_float(bits);
}

// Two E2M1 codes (one byte, element 0 in the low nibble) -> two fp32 values (exact).
__device__ __forceinline__ float2 e2m1x2_value(uint32_t byte)
{
    uint32_t h;
    uint16_t in = (uint16_t)(byte & 0xffu);
    asm("{\n\t.reg .b8 t;\n\tcvt.u8.u16 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}" : "=r"(h) : "h"(in));
    return __half22float2(*reinterpret_cast<__half2*>(&h));
}

// The per-block encode factor fl(S_enc / sb), saturated at the largest finite binary32 value.
// The quotient overflows only when S_enc itself was clamped there (tensor amax below
// 2688 / FLT_MAX, about 7.9e-36) and sb < 1; saturating keeps every product x * e_b finite, so
// x = 0 still encodes as a signed zero, as S_enc's own clamp does for the tensor scale.
__device__ __forceinline__ float encode_factor(float s_enc, float sbv)
{
    return fminf(__fdiv_rn(s_enc, sbv), 3.4028234663852886e38f);
}

// Quantization of one 16-element block held as 8 bf16x2 words.  Returns the scale byte,
// writes the 8 code bytes into code_lo / code_hi (element 2i in the low nibble of byte i).
struct BlockOut {
    uint32_t code_lo, code_hi;
    uint32_t sb;
    float e_b;  // fl(S_enc / sb) (unused when sb == 0)
    float d_b;  // fl(sb * S_dec)
};

__device__ __forceinline__ float block_amax(const float* v)
{
    float a = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(v[i]));
    return a;
}

__device__ __forceinline__ BlockOut quantize16(const float* v, float s_enc, float s_dec)
{
    BlockOut o;
    float amax_b = block_amax(v);
    float t = __fmul_rn(__fdiv_rn(amax_b, 6.0f), s_enc);
    o.sb = e4m3(t);
    float sbv = e4m3_value(o.sb);
    o.e_b = (o.sb == 0) ? 0.0f : encode_factor(s_enc, sbv);
    o.d_b = __fmul_rn(sbv, s_dec);
    uint32_t c[8];
    if (o.sb == 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            c[i] = ((__float_as_uint(v[2 * i]) >> 28) & 0x8u) | ((__float_as_uint(v[2 * i + 1]) >> 24) & 0x80u);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) c[i] = e2m1x2(__fmul_rn(v[2 * i], o.e_b), __fmul_rn(v[2 * i + 1], o.e_b));
    }
    o.code_lo = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
    o.code_hi = c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24);
    return o;
}

// Residual r = fl(x - fl(V[q] * d_b)).
__device__ __forceinline__ float residual(float x, uint32_t code, float d_b)
{
    return __fsub_rn(x, __fmul_rn(e2m1_value(code), d_b));
}

// Score term of one residual: q = rint(|r| * 2^(20 - E)), returned squared.  `sc` is 2^(20-E)
// when that power is a normal float; otherwise sc_a * sc_b split it (both powers of two).
struct ScoreScale {
    float sc_a, sc_b;
    bool split;
};

__device__ __forceinline__ ScoreScale score_scale(int32_t shift_e)
{
    ScoreScale s;
    int p = 20 - shift_e;
    if (p >= -126 && p <= 127) {
        s.sc_a = __uint_as_float((uint32_t)(p + 127) << 23);
        s.sc_b = 1.0f;
        s.split = false;
    } else {
        int pa = p / 2, pb = p - pa;
        s.sc_a = __uint_as_float((uint32_t)(pa + 127) << 23);
        s.sc_b = __uint_as_float((uint32_t)(pb + 127) << 23);
        s.split = true;
    }
    return s;
}

__device__ __forceinline__ uint64_t score_term(float r, const ScoreScale& s)
{
    // |r| * 2^p < 2^19, so adding 2^23 leaves the rounded integer in the low mantissa bits.
    float a = fabsf(r);
    if (s.split) a = __fmul_rn(a, s.sc_a);
    float y = __fmaf_rn(a, s.split ? s.sc_b : s.sc_a, 8388608.0f);
    uint32_t q = __float_as_uint(y) & 0x7fffffu;
    return (uint64_t)q * (uint64_t)q;
}

// The first error a kernel records in the device status word wins; `where` identifies the
// site (a wait or a check).
__device__ __forceinline__ void report_status(DeviceStatus* st, nvq_status code, int where)
{
    if (atomicCAS(&st->status, 0, (int)code) == 0) atomicExch(&st->where, where);
}

// ------------------------------------------------------------------ packed fp32 pairs
// Two binary32 values in one 64-bit register (low word = first element), for the paired FP32
// instructions of sm_100+ (one instruction, two independently rounded results).
__device__ __forceinline__ uint64_t f2pack(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f2unpack(uint64_t v, float& lo, float& hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// bf16x2 word -> fp32 pair (exact).
__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t w) { return f2pack(bf16lo(w), bf16hi(w)); }

__device__ __forceinline__ uint64_t f2mul(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t f2add(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t f2sub(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// Bounded mbarrier / flag waits record this in the device status word.
__device__ __forceinline__ void report_timeout(DeviceStatus* st, int where) { report_status(st, NVQ_ERR_TIMEOUT, where); }

// A channel index read from a caller's selection list (idx): inside [0, K) it is returned as
// is; outside, the device status records NVQ_ERR_ARG at `where` and channel 0 is used instead,
// so that no load leaves the operand (the call's output is then meaningless, and the status
// says so).  One unsigned compare per index.
constexpr int kWhereBadChannelAct = 42;     // act_tail_kernel / row_tail_kernel<true>
constexpr int kWhereBadChannelWeight = 43;  // weight tails
constexpr int kWhereBadChannelRecon = 44;   // rac_reconstruct
__device__ __forceinline__ int checked_channel(int j, int K, DeviceStatus* st, int where)
{
    if ((unsigned)j >= (unsigned)K) {
        report_status(st, NVQ_ERR_ARG, where);
        return 0;
    }
    return j;
}

// The same check for unrolled gather loops, without a branch: an index outside [0, K) becomes
// channel 0 and sets `bad`, which the caller reports once after the loop (a branch and an
// atomic per index would hold every load of the loop behind its own check).
__device__ __forceinline__ int clamp_channel(int j, int K, bool& bad)
{
    const bool out = (unsigned)j >= (unsigned)K;
    bad |= out;
    return out ? 0 : j;
}

// Bound of the wait, after another wait of the CTA ran out, for the asynchronous copies it
// already issued to land before it exits (they complete within microseconds; this bound does
// not shrink with the configurable limit, so even a tiny limit never lets a CTA exit while a
// copy into its shared memory is in flight).
constexpr unsigned long long kDrainWaitCycles = 1ull << 26;
__host__ __device__ __forceinline__ unsigned long long drain_limit(unsigned long long limit)
{
    return limit > kDrainWaitCycles ? limit : kDrainWaitCycles;
}

}  // namespace nvq
