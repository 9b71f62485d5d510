// fp8.cu -- the quantizer of the FP8 W8A8 baseline the paper compares against (QUADS §2.2
// "FP8": E4M3 elements, every tile of values carrying its own scale, as DeepGEMM does; §4.4.2:
// FP8 W8A8 rollout is the production baseline).
//
// Tiles: 1 x 128 for activations (one row, 128 consecutive channels), 128 x 128 for weights.
// Tile scale alpha = 2^e, e the smallest integer with 448 * 2^e >= amax of the tile, clamped to
// [-127, 127] (an all-zero tile gets -127), stored as the UE8M0 byte e + 127 in the blocked scale
// layout the block-scaled MMA reads with one scale per 32 elements (scale_vec::1X): a tile's
// byte fills its 4 scale columns (and, for weights, its 128 rows).  Element: E4M3 of x * 2^-e,
// nearest, ties to even, sign kept; |x * 2^-e| <= 448, and the scaling by a power of two is exact.
//
//   fp8_act_kernel     half-warp per 1 x 128 tile: one 16-byte load of 8 elements per lane,
//                      the tile amax by shuffles inside the half-warp, 8 code bytes per lane.
//   fp8_weight_kernel  CTA per 128 x 128 tile: 64 elements per thread held in registers, the
//                      amax by the CTA, then the codes; the scale word of each of the 128 rows.
#include <cuda_bf16.h>

#include "common.cuh"

namespace nvq {

// e of the tile scale from amax >= 0.  With amax = 1.m * 2^E and 448 = 1.75 * 2^8,
// 448 * 2^e >= amax  <=>  e >= E - 8 + [1.m > 1.75]; zero and subnormal amax lie below 448 * 2^-127.
__device__ __forceinline__ int fp8_tile_exponent(float amax)
{
    const uint32_t u = __float_as_uint(amax);
    const int ef = (int)(u >> 23);
    if (ef == 0) return -127;
    const int e = ef - 127 - 8 + ((u & 0x7fffffu) > 0x600000u ? 1 : 0);
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^-e as a float (e in [-127, 126]: always a normal power of two).
__device__ __forceinline__ float pow2_neg(int e) { return __uint_as_float((uint32_t)(127 - e) << 23); }

// Two fp32 -> two E4M3 bytes (lo -> low byte), nearest even, saturating, sign kept.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Eight bf16 (one 16-byte word) times s -> eight E4M3 bytes.
__device__ __forceinline__ uint2 encode8(const uint4& v, float s)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t b[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) b[i] = e4m3x2(__fmul_rn(bf16lo(w[i]), s), __fmul_rn(bf16hi(w[i]), s));
    return make_uint2(b[0] | (b[1] << 16), b[2] | (b[3] << 16));
}

__device__ __forceinline__ float amax8(const uint4& v)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) m = fmaxf(m, fmaxf(fabsf(bf16lo(w[i])), fabsf(bf16hi(w[i]))));
    return m;
}

// The scale word of columns 4t .. 4t+3 of one row: the tile byte on the columns below K / 32.
__device__ __forceinline__ uint32_t scale_word(int e, int t, int K)
{
    const int valid = K / 32 - 4 * t;  // 1..4
    const uint32_t b = (uint32_t)(e + 127);
    uint32_t w = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        if (i < valid) w |= b << (8 * i);
    return w;
}

__global__ void __launch_bounds__(256) fp8_act_kernel(const __nv_bfloat16* __restrict__ x, int64_t ldx, int64_t rows, int K,
                                                      uint8_t* __restrict__ codes, int64_t ld_codes, uint8_t* __restrict__ sf,
                                                      int64_t sf_cols)
{
    const int tiles_per_row = (K + 127) / 128;
    const int64_t tile = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 4;
    const int l = threadIdx.x & 15;
    // every lane takes part in the shuffles; lanes past the end or past K hold zeros
    const bool live = tile < rows * tiles_per_row;
    const int64_t r = live ? tile / tiles_per_row : 0;
    const int t = live ? (int)(tile - r * tiles_per_row) : 0;
    const int c = t * 128 + l * 8;  // K % 32 == 0: c < K means all 8 elements are inside
    const bool has = live && c < K;
    const uint4 v = has ? __ldg(reinterpret_cast<const uint4*>(x + r * ldx + c)) : make_uint4(0, 0, 0, 0);
    float m = amax8(v);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const int e = fp8_tile_exponent(m);
    if (has) *reinterpret_cast<uint2*>(codes + r * ld_codes + c) = encode8(v, pow2_neg(e));
    if (live && l == 0) *reinterpret_cast<uint32_t*>(sf + sf_offset(r, 4 * t, sf_cols)) = scale_word(e, t, K);
}

constexpr int kWTile = 128;
constexpr int kWThreads = 256;
constexpr int kWRowsPerPass = kWThreads / 16;        // 16 threads x 8 elements cover a row of the tile
constexpr int kWPasses = kWTile / kWRowsPerPass;     // 8

__global__ void __launch_bounds__(kWThreads) fp8_weight_kernel(const __nv_bfloat16* __restrict__ x, int64_t ldx,
                                                               int64_t rows, int K, uint8_t* __restrict__ codes,
                                                               int64_t ld_codes, uint8_t* __restrict__ sf, int64_t sf_cols)
{
    __shared__ float warp_max[kWThreads / 32];
    const int t = blockIdx.y;                        // column tile
    const int64_t r0 = (int64_t)blockIdx.x * kWTile;  // first row of the tile
    const int tid = threadIdx.x;
    const int c = t * 128 + (tid & 15) * 8;
    const bool col_ok = c < K;
    uint4 v[kWPasses];
    float m = 0.0f;
#pragma unroll
    for (int p = 0; p < kWPasses; ++p) {
        const int64_t r = r0 + p * kWRowsPerPass + (tid >> 4);
        v[p] = (col_ok && r < rows) ? __ldg(reinterpret_cast<const uint4*>(x + r * ldx + c)) : make_uint4(0, 0, 0, 0);
        m = fmaxf(m, amax8(v[p]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((tid & 31) == 0) warp_max[tid >> 5] = m;
    __syncthreads();
    m = 0.0f;
#pragma unroll
    for (int i = 0; i < kWThreads / 32; ++i) m = fmaxf(m, warp_max[i]);
    const int e = fp8_tile_exponent(m);
    const float s = pow2_neg(e);
#pragma unroll
    for (int p = 0; p < kWPasses; ++p) {
        const int64_t r = r0 + p * kWRowsPerPass + (tid >> 4);
        if (col_ok && r < rows) *reinterpret_cast<uint2*>(codes + r * ld_codes + c) = encode8(v[p], s);
    }
    if (tid < kWTile && r0 + tid < rows)
        *reinterpret_cast<uint32_t*>(sf + sf_offset(r0 + tid, 4 * t, sf_cols)) = scale_word(e, t, K);
}

}  // namespace nvq

using namespace nvq;

extern "C" int64_t nvq_fp8_sf_cols(int64_t K) { return ((K / 32) + 3) / 4 * 4; }

extern "C" nvq_status fp8_quantize(const void* x, int64_t rows, int64_t K, int64_t ldx, int32_t tile_rows, uint8_t* codes,
                                   int64_t ld_codes, uint8_t* sf, int64_t sf_cols, void* stream)
{
    NVQ_TRACE("fp8_quantize");
    static const char* fn = "fp8_quantize";
    NVQ_CHECK_ARG(x && codes && sf, NVQ_ERR_ARG, "%s: null pointer argument", fn);
    NVQ_CHECK_ARG(tile_rows == 1 || tile_rows == 128, NVQ_ERR_ARG, "%s: tile_rows must be 1 or 128", fn);
    NVQ_CHECK_ARG(rows >= 1 && rows <= (1ll << 24), NVQ_ERR_SHAPE, "%s: rows outside [1, 2^24]", fn);
    NVQ_CHECK_ARG(K >= 32 && K <= 16384 && K % 32 == 0, NVQ_ERR_SHAPE, "%s: K must be a multiple of 32 in [32, 16384]", fn);
    NVQ_CHECK_ARG(sf_cols >= nvq_fp8_sf_cols(K) && sf_cols % 4 == 0, NVQ_ERR_SHAPE, "%s: sf_cols must be >= nvq_fp8_sf_cols(K)", fn);
    NVQ_CHECK_ARG(ldx >= K && ldx % 8 == 0 && aligned(x, 16) && ld_codes >= K && ld_codes % 16 == 0 && aligned(codes, 16) &&
                      aligned(sf, 4),
                  NVQ_ERR_ALIGN, "%s: rows of x and codes must be 16-byte aligned", fn);
    set_error("");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const auto* xb = static_cast<const __nv_bfloat16*>(x);
    if (tile_rows == 1) {
        const int64_t threads = rows * ((K + 127) / 128) * 16;
        fp8_act_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(xb, ldx, rows, (int)K, codes, ld_codes, sf, sf_cols);
        NVQ_LAUNCH_CHECK("fp8_act_kernel");
    } else {
        const dim3 grid((unsigned)((rows + kWTile - 1) / kWTile), (unsigned)((K + 127) / 128));
        fp8_weight_kernel<<<grid, kWThreads, 0, st>>>(xb, ldx, rows, (int)K, codes, ld_codes, sf, sf_cols);
        NVQ_LAUNCH_CHECK("fp8_weight_kernel");
    }
    return NVQ_OK;
}
