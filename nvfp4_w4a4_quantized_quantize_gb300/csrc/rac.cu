// rac.cu -- Residual Activation Compensation (QUADS §3.3).
//
//   topk_kernel            S = TopK of the channel scores (Eq. (24)), one CTA per group: an
//                          MSB-first radix select over the uint64 scores finds the k-th largest
//                          score (stopping once its bin holds exactly the channels still
//                          needed), ties at the threshold go to the lower channel index, and a
//                          block scan emits the selected channels in ascending order.
//   act_tail_kernel        second pass of Eq. (21): the residual X - DQ(Q(X)) on the selected
//                          channels (recomputed from x and the stored block scale,
//                          bit-identical to the first pass) is quantized, 16 selected channels
//                          per block, into the tail columns [K, K + k) of the activation operand.
//   weight_tail_kernel     the weight columns that multiply the correction: dequantized stored
//                          weights on the selected channels, re-quantized with the weight's
//                          S_enc, into the tail columns of the weight operand (gathered from
//                          the row-major operand);
//   weight_tail_cm_kernel  the same tail from a channel-major copy of the weights
//                          (channel_major_codes_kernel / channel_major_sf_kernel make it);
//   row_tail_kernel        both tails for a large share of channels: whole rows expanded in
//                          shared memory, then gathered (the schedule nvq_set_tail_path picks).
#include <cuda_bf16.h>

#include "common.cuh"

namespace nvq {

static constexpr int kTopkThreads = 1024;

// Exclusive scan of one int per thread over the block; returns the block total in *total.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_sums, int* total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int s = (lane < (int)(blockDim.x >> 5)) ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        warp_sums[lane] = s;  // inclusive
    }
    __syncthreads();
    int base = (warp == 0) ? 0 : warp_sums[warp - 1];
    *total = warp_sums[(blockDim.x >> 5) - 1];
    __syncthreads();
    return base + x - v;
}

// Radix select of the k-th largest score, MSB first, 8 bits per pass.  Every thread keeps its
// (at most 8) channels' scores in registers; per pass each warp folds equal digits with
// __match_any_sync before one shared atomic per distinct digit, so the histogram sees no
// contention.  The select stops as soon as the bin holding the k-th largest score holds exactly
// the channels still needed (usually after two or three passes): every channel whose decided
// high bits are above the prefix, and every channel of that bin, is taken.  Otherwise it runs to
// the last bit and the threshold T is exact; channels above T are all taken and the
// lowest-index channels equal to T fill the rest (ties to the lower channel index).
static constexpr int kTopkPer = 8;  // channels per thread: K <= 8192

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(const unsigned long long* __restrict__ scores, int K, int k,
                                                             int32_t* __restrict__ idx)
{
    __shared__ unsigned int hist2[2][256];
    __shared__ int warp_sums[32];
    __shared__ unsigned long long s_prefix, s_or;
    __shared__ int s_remaining, s_done;
    const int g = blockIdx.x;
    const unsigned long long* src = scores + (int64_t)g * K;
    int32_t* out = idx + (int64_t)g * k;
    const int tid = threadIdx.x, lane = tid & 31;
    const int per = (K + kTopkThreads - 1) / kTopkThreads;
    const int j0 = tid * per;
    unsigned long long key[kTopkPer];
    unsigned long long orv = 0;
#pragma unroll
    for (int q = 0; q < kTopkPer; ++q) {
        const int j = j0 + q;
        key[q] = (q < per && j < K) ? src[j] : 0ull;
        orv |= key[q];
    }
    if (tid == 0) { s_or = 0; s_prefix = 0; s_remaining = k; s_done = 0; }
    __syncthreads();
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) orv |= __shfl_xor_sync(0xffffffffu, orv, o);
    if (lane == 0 && orv) atomicOr(&s_or, orv);
    __syncthreads();
    const int top_bit = s_or ? 63 - __clzll(s_or) : 0;
    unsigned long long mask = 0;
    if (tid < 256) hist2[0][tid] = 0;
    __syncthreads();
    int par = 0;
    for (int shift = (top_bit / 8) * 8; shift >= 0; shift -= 8, par ^= 1) {
        unsigned int* hist = hist2[par];
        if (tid < 256) hist2[par ^ 1][tid] = 0;  // the next pass's histogram
        const unsigned long long prefix = s_prefix;
#pragma unroll
        for (int q = 0; q < kTopkPer; ++q) {
            if (q >= per) break;  // uniform across the block
            const int j = j0 + q;
            const int d = (j < K && (key[q] & mask) == prefix) ? (int)((key[q] >> shift) & 255u) : 256;
            const unsigned peers = __match_any_sync(0xffffffffu, d);
            if (d < 256 && lane == __ffs(peers) - 1) atomicAdd(&hist[d], (unsigned)__popc(peers));
        }
        __syncthreads();
        if (tid < 32) {
            // lane l owns digits 255-8l .. 248-8l (descending)
            int cnt[8], tot = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) { cnt[i] = (int)hist[255 - 8 * tid - i]; tot += cnt[i]; }
            int incl = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (tid >= o) incl += y;
            }
            int above = incl - tot;
            const int rem = s_remaining;
            __syncwarp();  // every lane has read s_remaining before the one owner lane rewrites it
            if (above < rem && rem <= incl) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (above < rem && rem <= above + cnt[i]) {
                        s_prefix = prefix | ((unsigned long long)(255 - 8 * tid - i) << shift);
                        s_remaining = rem - above;
                        s_done = cnt[i] == rem - above;  // the whole bin is needed
                    }
                    above += cnt[i];
                }
            }
        }
        mask |= 255ull << shift;
        __syncthreads();
        if (s_done) break;  // uniform: read after the barrier
    }
    // compare on the decided bits (all of them unless the select stopped early)
#pragma unroll
    for (int q = 0; q < kTopkPer; ++q) key[q] &= mask;
    const unsigned long long T = s_prefix;
    const int take_eq = s_remaining;
    int n_eq = 0;
#pragma unroll
    for (int q = 0; q < kTopkPer; ++q)
        if (q < per && j0 + q < K) n_eq += (key[q] == T);
    int total;
    const int eq_rank = block_exclusive_scan(n_eq, warp_sums, &total);
    int n_sel = 0;
    {
        int r = eq_rank;
#pragma unroll
        for (int q = 0; q < kTopkPer; ++q) {
            if (q >= per || j0 + q >= K) continue;
            const bool sel = key[q] > T || (key[q] == T && r < take_eq);
            r += (key[q] == T);
            n_sel += sel;
        }
    }
    int pos = block_exclusive_scan(n_sel, warp_sums, &total);
    {
        int r = eq_rank;
#pragma unroll
        for (int q = 0; q < kTopkPer; ++q) {
            if (q >= per || j0 + q >= K) continue;
            const bool sel = key[q] > T || (key[q] == T && r < take_eq);
            r += (key[q] == T);
            if (sel) out[pos++] = j0 + q;
        }
    }
}

// ------------------------------------------------------------------------ activation tail
// Thread per (row of a 64-row tile, share of the k/16 tail blocks): bsplit threads split a
// row's blocks (1 when there are rows enough to fill the GPU, more for short inputs).  The CTA stages
// the tile's group's selected channels and, for each of the 128 E4M3 scale codes, the encode
// factor fl(S_enc / sb) and decode factor fl(sb * S_dec) (the tables the first pass used), so a
// thread recomputes each gathered element's code and residual (bit-identical to the first
// pass) with lookups instead of divisions; it then quantizes each block of 16 residuals and
// writes its row's whole tail at once.  Rows of another group than the tile's first row (only
// with groups that do not start on 64-row boundaries) compute the factors directly.
constexpr int kTailRows = 64;

// A gathered bf16 element, its L2 line marked evict-first: after the tail the activation is
// not read again, so whatever the quantize pass kept in L2 for the tail is released.
__device__ __forceinline__ float ld_bf16_last_use(const __nv_bfloat16* p, uint64_t pol)
{
    unsigned short v;
    asm volatile("ld.global.nc.L2::cache_hint.b16 %0, [%1], %2;" : "=h"(v) : "l"(p), "l"(pol));
    return __uint_as_float((uint32_t)v << 16);
}

__global__ void __launch_bounds__(512) act_tail_kernel(const __nv_bfloat16* __restrict__ x, int64_t ldx, int K, int k,
                                                       Groups gr, const nvq_tensor_scale* __restrict__ ts,
                                                       const int32_t* __restrict__ idx, uint8_t* __restrict__ codes,
                                                       int64_t ld_codes, uint8_t* __restrict__ sf, int64_t sf_cols, int bsplit,
                                                       DeviceStatus* dst)
{
    __shared__ float eb_tab[128], db_tab[128];
    __shared__ int s_sel[512];
    __shared__ int s_g0;
    const int tid = threadIdx.x;
    const int t = tid % kTailRows;   // row in the tile
    const int part = tid / kTailRows;  // share of the row's blocks: b = part, part + bsplit, ...
    const int64_t tile_row = (int64_t)blockIdx.x * kTailRows;
    if (tid == 0) s_g0 = tile_row < gr.total_rows ? group_of_row(gr, tile_row) : 0;
    __syncthreads();
    const int g0 = s_g0;
    const float s_enc0 = ts[g0].s_enc, s_dec0 = ts[g0].s_dec;
    for (int e = tid; e < 128; e += blockDim.x) {
        const float sbv = e4m3_value((uint32_t)e);
        eb_tab[e] = (e == 0 || e == 127) ? 0.0f : encode_factor(s_enc0, sbv);
        db_tab[e] = (e == 127) ? 0.0f : __fmul_rn(sbv, s_dec0);
    }
    const bool sel_smem = k <= 512;  // larger channel sets are read from global memory
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    if (sel_smem)
        for (int c = tid; c < k; c += blockDim.x) s_sel[c] = checked_channel(idx[(int64_t)g0 * k + c], K, dst, kWhereBadChannelAct);
    __syncthreads();

    const int64_t row = tile_row + t;
    if (row >= gr.total_rows) return;
    int g = g0;
    if (gr.off != nullptr)
        while (g + 1 < gr.G && gr.off[g + 1] <= row) ++g;
    else
        g = group_of_row(gr, row);
    int64_t gb, ge;
    group_range(gr, g, gb, ge);
    if (row < gb || row >= ge) return;
    const bool own = g == g0;
    const float s_enc = own ? s_enc0 : ts[g].s_enc, s_dec = own ? s_dec0 : ts[g].s_dec;
    const int32_t* sel_g = idx + (int64_t)g * k;
    const __nv_bfloat16* xr = x + row * ldx;
    uint8_t* crow = codes + row * ld_codes + K / 2;
    const int nsb = K / 16;
    const bool word_sf = (nsb % 4) == 0 && bsplit == 1;
    uint32_t sfw = 0;
    bool bad = false;
    for (int b = part; b < k / 16; b += bsplit) {
        float xv[16];
        uint32_t sb[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int j = (own && sel_smem) ? s_sel[b * 16 + i] : clamp_channel(sel_g[b * 16 + i], K, bad);
            xv[i] = ld_bf16_last_use(xr + j, pol);
            sb[i] = sf[sf_offset(row, j >> 4, sf_cols)];
        }
        float rv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float e_b, d_b;
            if (own) {
                e_b = eb_tab[sb[i]];
                d_b = db_tab[sb[i]];
            } else {
                const float sbv = e4m3_value(sb[i]);
                e_b = sb[i] == 0 ? 0.0f : encode_factor(s_enc, sbv);
                d_b = __fmul_rn(sbv, s_dec);
            }
            const uint32_t code = e2m1x2(__fmul_rn(xv[i], e_b), 0.0f) & 0xfu;  // e_b 0: +-0 keeps the sign
            rv[i] = residual(xv[i], code, d_b);
        }
        const BlockOut o = quantize16(rv, s_enc, s_dec);
        *reinterpret_cast<uint2*>(crow + 8 * b) = make_uint2(o.code_lo, o.code_hi);
        if (word_sf) {
            sfw |= o.sb << (8 * (b & 3));
            if ((b & 3) == 3) {
                *reinterpret_cast<uint32_t*>(sf + sf_offset(row, nsb + b - 3, sf_cols)) = sfw;
                sfw = 0;
            }
        } else {
            sf[sf_offset(row, nsb + b, sf_cols)] = (uint8_t)o.sb;
        }
    }
    if (bad) report_status(dst, NVQ_ERR_ARG, kWhereBadChannelAct);
    const int64_t c0 = (K + k) / 16;
    if (word_sf && (c0 & 3)) {
        *reinterpret_cast<uint32_t*>(sf + sf_offset(row, c0 & ~3ll, sf_cols)) = sfw;  // rest of the group: padding
        for (int64_t c = (c0 | 3) + 1; c < sf_cols; ++c) sf[sf_offset(row, c, sf_cols)] = 0;
    } else if (part == 0) {
        for (int64_t c = c0; c < sf_cols; ++c) sf[sf_offset(row, c, sf_cols)] = 0;
    }
}

// ------------------------------------------------------------------------ weight tail
// Thread per (weight row, tail block).  Weight rows of group g are [g * N, (g + 1) * N).
__global__ void __launch_bounds__(256) weight_tail_kernel(uint8_t* __restrict__ codes, int64_t ld_codes,
                                                           uint8_t* __restrict__ sf, int64_t sf_cols, int64_t N, int K,
                                                           int k, int G, const nvq_tensor_scale* __restrict__ ts,
                                                           const int32_t* __restrict__ idx, int idx_per_group,
                                                           DeviceStatus* dst)
{
    const int nbt = k / 16;
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t total = (int64_t)G * N * nbt;
    if (t >= total) return;
    const int b = (int)(t % nbt);
    const int64_t row = t / nbt;
    const int g = (int)(row / N);
    const float s_enc = ts[g].s_enc, s_dec = ts[g].s_dec;
    const int32_t* sel = idx + (idx_per_group ? (int64_t)g * k : 0);
    const uint8_t* cr = codes + row * ld_codes;
    bool bad = false;
    float wv[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int j = clamp_channel(sel[b * 16 + i], K, bad);
        const uint32_t c = (cr[j >> 1] >> ((j & 1) * 4)) & 0xfu;
        const uint32_t sb = sf[sf_offset(row, j >> 4, sf_cols)];
        wv[i] = __fmul_rn(e2m1_value(c), __fmul_rn(e4m3_value(sb), s_dec));
    }
    if (bad) report_status(dst, NVQ_ERR_ARG, kWhereBadChannelWeight);
    BlockOut o = quantize16(wv, s_enc, s_dec);
    *reinterpret_cast<uint2*>(codes + row * ld_codes + (K + 16 * b) / 2) = make_uint2(o.code_lo, o.code_hi);
    sf[sf_offset(row, K / 16 + b, sf_cols)] = (uint8_t)o.sb;
    if (b == 0)
        for (int64_t c = (K + k) / 16; c < sf_cols; ++c) sf[sf_offset(row, c, sf_cols)] = 0;
}

// Same tail from the channel-major copy (nvfp4_channel_major): CTA per (group, 64 weight rows,
// chunk of up to 256 selected channels), split threads per row (1, 2 or 4: the tail blocks of
// a row are dealt round-robin to them).  The CTA first stages, for each channel of its chunk,
// the 32 code bytes and 64 scale bytes of its rows into shared memory with 16-byte loads (all
// in flight together); then each thread builds its blocks of its row from there: 8 code bytes
// and the scale byte per block.  The thread holding a row's last tail block of the last chunk
// also zeroes the row's scale padding.
constexpr int kWtRows = 64;
constexpr int kWtChunk = 256;  // selected channels staged per pass (24 KB of shared memory)
constexpr int kWtMaxSplit = 4;

// quantize16 with the encode factor fl(S_enc / sb) read from a per-group table (eb_tab[sb],
// 0 for sb = 0) instead of divided per block: the same scale byte and codes.
__device__ __forceinline__ void quantize16_tab(const float* v, float s_enc, const float* eb_tab, uint32_t& sb,
                                               uint32_t& code_lo, uint32_t& code_hi)
{
    const float amax_b = block_amax(v);
    sb = e4m3(__fmul_rn(__fdiv_rn(amax_b, 6.0f), s_enc));
    const float e_b = eb_tab[sb];
    uint32_t c[8];
    if (sb == 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            c[i] = ((__float_as_uint(v[2 * i]) >> 28) & 0x8u) | ((__float_as_uint(v[2 * i + 1]) >> 24) & 0x80u);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) c[i] = e2m1x2(__fmul_rn(v[2 * i], e_b), __fmul_rn(v[2 * i + 1], e_b));
    }
    code_lo = c[0] | (c[1] << 8) | (c[2] << 16) | (c[3] << 24);
    code_hi = c[4] | (c[5] << 8) | (c[6] << 16) | (c[7] << 24);
}

__global__ void __launch_bounds__(kWtRows * kWtMaxSplit) weight_tail_cm_kernel(
    uint8_t* __restrict__ codes, int64_t ld_codes, uint8_t* __restrict__ sf, int64_t sf_cols, int64_t N, int K, int k,
    const nvq_tensor_scale* __restrict__ ts, const int32_t* __restrict__ idx, int idx_per_group,
    const uint8_t* __restrict__ cm_codes, const uint8_t* __restrict__ cm_sf, DeviceStatus* dst)
{
    extern __shared__ __align__(16) uint8_t wt_smem[];
    // per-group tables: E2M1 values, dequantization scale fl(sb * S_dec) and encode factor
    // fl(S_enc / sb) of every E4M3 scale byte (the same operations as the direct forms)
    __shared__ float v_tab[16], db_tab[128], eb_tab[128];
    const int kc = k < kWtChunk ? k : kWtChunk;   // channels staged at a time
    uint8_t* s_codes = wt_smem;                    // [kc][32]: rows n0 .. n0+63, two per byte
    uint8_t* s_sf = wt_smem + (size_t)kc * 32;     // [kc][64]
    const int c0 = blockIdx.z * kWtChunk;
    const int g = blockIdx.y;
    const int64_t n0 = (int64_t)blockIdx.x * kWtRows;
    const int nthr = blockDim.x;
    const int split = nthr / kWtRows;
    const int t = threadIdx.x % kWtRows;   // row in the tile
    const int part = threadIdx.x / kWtRows;
    const int nsb = K / 16;
    const int32_t* sel = idx + (idx_per_group ? (int64_t)g * k : 0);
    const float s_enc = ts[g].s_enc, s_dec = ts[g].s_dec;
    const int64_t row = (int64_t)g * N + n0 + t;
    uint8_t* crow = codes + row * ld_codes + K / 2;
    const int cnt = k - c0 < kc ? k - c0 : kc;  // channels of this chunk (a multiple of 16)
    for (int e = threadIdx.x; e < 128; e += nthr) {
        const float sbv = e4m3_value((uint32_t)e);
        db_tab[e] = __fmul_rn(sbv, s_dec);
        eb_tab[e] = e == 0 ? 0.0f : encode_factor(s_enc, sbv);
        if (e < 16) v_tab[e] = e2m1_value((uint32_t)e);
    }
    // stage: per channel 2 x 16 code bytes + 4 x 16 scale bytes
    for (int w = threadIdx.x; w < cnt * 6; w += nthr) {
        const int c = w / 6, q = w % 6;
        const int j = checked_channel(sel[c0 + c], K, dst, kWhereBadChannelWeight);
        uint4 v;
        if (q < 2)
            v = __ldg(reinterpret_cast<const uint4*>(cm_codes + ((int64_t)g * K + j) * (N / 2) + n0 / 2) + q);
        else
            v = __ldg(reinterpret_cast<const uint4*>(cm_sf + ((int64_t)g * nsb + (j >> 4)) * N + n0) + (q - 2));
        if (q < 2) reinterpret_cast<uint4*>(s_codes + c * 32)[q] = v;
        else reinterpret_cast<uint4*>(s_sf + c * 64)[q - 2] = v;
    }
    __syncthreads();
    const int b_end = (c0 + cnt) / 16;
    for (int b = c0 / 16 + part; b < b_end; b += split) {
        float wv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int c = b * 16 + i - c0;
            const uint32_t code = (s_codes[c * 32 + (t >> 1)] >> ((t & 1) * 4)) & 0xfu;
            const uint32_t sb = s_sf[c * 64 + t] & 0x7fu;
            wv[i] = __fmul_rn(v_tab[code], db_tab[sb]);  // fl(V[q] * fl(sb * S_dec))
        }
        uint32_t osb, lo, hi;
        quantize16_tab(wv, s_enc, eb_tab, osb, lo, hi);
        *reinterpret_cast<uint2*>(crow + 8 * b) = make_uint2(lo, hi);
        sf[sf_offset(row, nsb + b, sf_cols)] = (uint8_t)osb;
    }
    // scale padding of the row: by the thread that holds the row's last tail block
    if (c0 + kWtChunk < k || part != (b_end - 1 - c0 / 16) % split) return;
    for (int64_t c = (K + k) / 16; c < sf_cols; ++c) sf[sf_offset(row, c, sf_cols)] = 0;
}

// Channel-major copy of the codes: CTA per (group, 64 rows, 128 channels) tile, transposed
// through shared memory.  Out byte (g, j, m) packs channel j of rows 2m (low nibble) and 2m + 1.
__global__ void __launch_bounds__(256) channel_major_codes_kernel(const uint8_t* __restrict__ codes, int64_t ld_codes,
                                                                   int64_t N, int K, uint8_t* __restrict__ cm_codes)
{
    __shared__ uint8_t tile[64][64 + 4];  // 64 rows x 64 bytes (128 channels)
    const int g = blockIdx.z;
    const int64_t n0 = (int64_t)blockIdx.y * 64;
    const int j0 = blockIdx.x * 128;
    const int tid = threadIdx.x;
    const int kb = K / 2;  // code bytes per row
    // load: 64 rows x 4 words of 16 bytes
    {
        const int r = tid >> 2, q = tid & 3;
        const int off = j0 / 2 + q * 16;
        const uint8_t* src = codes + ((int64_t)g * N + n0 + r) * ld_codes + off;
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (off + 16 <= kb) {
            const uint4 v = *reinterpret_cast<const uint4*>(src);
            w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
        } else {
            for (int i = 0; i < 16 && off + i < kb; ++i) w[i >> 2] |= (uint32_t)src[i] << (8 * (i & 3));
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) *reinterpret_cast<uint32_t*>(&tile[r][q * 16 + 4 * i]) = w[i];
    }
    __syncthreads();
    // store: channel j = j0 + tid / 2, bytes [16 h, 16 h + 16) of its 32-byte row segment
    const int jl = tid >> 1, h = tid & 1;
    const int j = j0 + jl;
    if (j >= K) return;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const int ra = 2 * (16 * h + m);
        const uint32_t lo = (tile[ra][jl >> 1] >> ((jl & 1) * 4)) & 0xfu;
        const uint32_t hi = (tile[ra + 1][jl >> 1] >> ((jl & 1) * 4)) & 0xfu;
        w[m >> 2] |= (lo | (hi << 4)) << (8 * (m & 3));
    }
    *reinterpret_cast<uint4*>(cm_codes + ((int64_t)g * K + j) * (N / 2) + n0 / 2 + 16 * h) = make_uint4(w[0], w[1], w[2], w[3]);
}

// Channel-major copy of the block scales: out byte (g, block c, row n), n fastest.
__global__ void __launch_bounds__(256) channel_major_sf_kernel(const uint8_t* __restrict__ sf, int64_t sf_cols, int64_t N,
                                                                int nsb, int G, uint8_t* __restrict__ cm_sf)
{
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= (int64_t)G * nsb * N) return;
    const int64_t n = t % N;
    const int64_t c = (t / N) % nsb;
    const int64_t g = t / (N * nsb);
    cm_sf[t] = sf[sf_offset(g * N + n, c, sf_cols)];
}

// ------------------------------------------------------------------------ row-path tails
// When S is a large share of K the kernels above spend their issue slots on one scattered load
// per selected element.  This one reads R whole rows with 16-byte loads, expands every channel's
// value into shared memory (fp32, one pad word after every 16 channels, so that lanes on
// neighbouring 16-channel blocks hit distinct banks), then gathers the selected channels from
// there and quantizes them into the tail:
//   kResidual   activations: the residual fl(x - fl(V * d_b)), the code recomputed from x and the
//               stored block scale exactly as the gather kernel does (bit-identical to the first pass);
//   !kResidual  weights: the dequantized stored weight fl(V * fl(sb * S_dec)).
constexpr int kRowThreads = 256;
constexpr int kRowElems = 8192;  // channels expanded per CTA: R = max(1, 8192 / K) rows

__host__ __device__ constexpr int row_tile_rows(int K) { return K >= kRowElems ? 1 : kRowElems / K; }
__host__ __device__ constexpr int padded_ch(int j) { return j + (j >> 4); }

inline size_t row_tail_smem(int K) { return (size_t)row_tile_rows(K) * (padded_ch(K) * sizeof(float) + sizeof(int)); }

template <bool kResidual>
__global__ void __launch_bounds__(kRowThreads)
    row_tail_kernel(const __nv_bfloat16* __restrict__ x, int64_t ldx, uint8_t* __restrict__ codes, int64_t ld_codes,
                    uint8_t* __restrict__ sf, int64_t sf_cols, int K, int k, Groups gr,
                    const nvq_tensor_scale* __restrict__ ts, const int32_t* __restrict__ idx, int idx_per_group,
                    int idx_vec, DeviceStatus* dst)
{
    extern __shared__ __align__(16) float rt_smem[];
    const int R = row_tile_rows(K);
    const int stride = padded_ch(K);
    int* s_g = reinterpret_cast<int*>(rt_smem + (size_t)R * stride);  // group of each row, -1: not written
    const int64_t row0 = (int64_t)blockIdx.x * R;
    const int tid = threadIdx.x;
    for (int r = tid; r < R; r += kRowThreads) {
        const int64_t row = row0 + r;
        int g = -1;
        if (row < gr.total_rows) {
            g = group_of_row(gr, row);
            int64_t b0, b1;
            group_range(gr, g, b0, b1);
            if (row < b0 || row >= b1) g = -1;
        }
        s_g[r] = g;
    }
    __syncthreads();
    // 1. expand: thread per (row, 16-channel block)
    const int nb = K / 16;
    for (int w = tid; w < R * nb; w += kRowThreads) {
        const int r = w / nb, b = w - r * nb;
        const int g = s_g[r];
        if (g < 0) continue;
        const int64_t row = row0 + r;
        const uint32_t sb = sf[sf_offset(row, b, sf_cols)];
        const float sbv = e4m3_value(sb);
        float* dst = rt_smem + (size_t)r * stride + padded_ch(16 * b);
        if constexpr (kResidual) {
            const float e_b = (sb == 0 || sb == 127) ? 0.0f : encode_factor(ts[g].s_enc, sbv);
            const float d_b = (sb == 127) ? 0.0f : __fmul_rn(sbv, ts[g].s_dec);
            const uint4* xp = reinterpret_cast<const uint4*>(x + row * ldx + 16 * b);
            const uint4 v0 = __ldg(xp), v1 = __ldg(xp + 1);
            const uint32_t xw[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float xa = bf16lo(xw[i]), xb = bf16hi(xw[i]);
                const float2 q = e2m1x2_value(e2m1x2(__fmul_rn(xa, e_b), __fmul_rn(xb, e_b)));
                dst[2 * i] = __fsub_rn(xa, __fmul_rn(q.x, d_b));
                dst[2 * i + 1] = __fsub_rn(xb, __fmul_rn(q.y, d_b));
            }
        } else {
            const float d_b = __fmul_rn(sbv, ts[g].s_dec);
            const uint2 c = *reinterpret_cast<const uint2*>(codes + row * ld_codes + 8 * b);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float2 q = e2m1x2_value(((i < 4 ? c.x : c.y) >> (8 * (i & 3))) & 0xffu);
                dst[2 * i] = __fmul_rn(q.x, d_b);
                dst[2 * i + 1] = __fmul_rn(q.y, d_b);
            }
        }
    }
    __syncthreads();
    // 2. gather + quantize: thread per (row, tail block)
    const int nbt = k / 16;
    for (int w = tid; w < R * nbt; w += kRowThreads) {
        const int r = w / nbt, b = w - r * nbt;
        const int g = s_g[r];
        if (g < 0) continue;
        const int64_t row = row0 + r;
        const int32_t* sel = idx + (idx_per_group ? (int64_t)g * k : 0) + 16 * b;
        int j[16];
        if (idx_vec) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int4 v = __ldg(reinterpret_cast<const int4*>(sel) + q);
                j[4 * q] = v.x; j[4 * q + 1] = v.y; j[4 * q + 2] = v.z; j[4 * q + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) j[i] = __ldg(sel + i);
        }
        bool bad = false;
#pragma unroll
        for (int i = 0; i < 16; ++i) j[i] = clamp_channel(j[i], K, bad);
        if (bad) report_status(dst, NVQ_ERR_ARG, kResidual ? kWhereBadChannelAct : kWhereBadChannelWeight);
        const float* src = rt_smem + (size_t)r * stride;
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = src[padded_ch(j[i])];
        const BlockOut o = quantize16(v, ts[g].s_enc, ts[g].s_dec);
        *reinterpret_cast<uint2*>(codes + row * ld_codes + K / 2 + 8 * b) = make_uint2(o.code_lo, o.code_hi);
        sf[sf_offset(row, nb + b, sf_cols)] = (uint8_t)o.sb;
        if (b == 0)
            for (int64_t c = (K + k) / 16; c < sf_cols; ++c) sf[sf_offset(row, c, sf_cols)] = 0;
    }
}

// Row path when the setting asks for it, or (NVQ_TAIL_AUTO) past the crossover measured on GB300
// at the MoE shapes: k >= K / 4 for activation tails and for weight tails gathered from the
// row-major operand.  A weight tail with the channel-major copy keeps its gather at every k (it
// reads only the selected channels' bytes, 16 at a time, and measured at or below the row path
// up to k = K).
inline bool use_row_tail(int K, int k, bool channel_major)
{
    if (tail_path() != NVQ_TAIL_AUTO) return tail_path() == NVQ_TAIL_ROWS;
    return !channel_major && 4 * k >= K;
}

template <bool kResidual>
nvq_status launch_row_tail(const void* x, int64_t ldx, uint8_t* codes, int64_t ld_codes, uint8_t* sf, int64_t sf_cols,
                           int K, int k, Groups gr, const nvq_tensor_scale* ts, const int32_t* idx, int idx_per_group,
                           cudaStream_t st)
{
    const int R = row_tile_rows(K);
    const int64_t tiles = (gr.total_rows + R - 1) / R;
    const int idx_vec = aligned(idx, 16) ? 1 : 0;  // per-group offsets g * k * 4 bytes keep 16-byte alignment
    DeviceStatus* dst = device_status_ptr();
    NVQ_CHECK_ARG(dst, NVQ_ERR_CUDA, "row tail: device status word unavailable");
    row_tail_kernel<kResidual><<<(unsigned)tiles, kRowThreads, row_tail_smem(K), st>>>(
        static_cast<const __nv_bfloat16*>(x), ldx, codes, ld_codes, sf, sf_cols, K, k, gr, ts, idx, idx_per_group, idx_vec,
        dst);
    NVQ_LAUNCH_CHECK(kResidual ? "row_tail_kernel<residual>" : "row_tail_kernel<weight>");
    return NVQ_OK;
}

nvq_status weight_tail_impl(uint8_t* codes, int64_t ld_codes, uint8_t* sf, int64_t sf_cols, int64_t N, int K, int k,
                            int G, const nvq_tensor_scale* ts, const int32_t* idx, int idx_per_group, cudaStream_t st)
{
    if (k == 0) return NVQ_OK;
    const int64_t total = (int64_t)G * N * (k / 16);
    const int threads = 256;
    DeviceStatus* dst = device_status_ptr();
    NVQ_CHECK_ARG(dst, NVQ_ERR_CUDA, "weight tail: device status word unavailable");
    weight_tail_kernel<<<(unsigned)((total + threads - 1) / threads), threads, 0, st>>>(
        codes, ld_codes, sf, sf_cols, N, K, k, G, ts, idx, idx_per_group, dst);
    NVQ_LAUNCH_CHECK("weight_tail_kernel");
    return NVQ_OK;
}

}  // namespace nvq

using namespace nvq;

static nvq_status check_rac_args(const char* fn, const void* x, int64_t rows, int64_t K, int64_t ldx,
                                 const int64_t* grp_off, int32_t groups, const nvq_tensor_scale* tscale, int32_t k,
                                 const uint8_t* codes, int64_t ld_codes, const uint8_t* sf, int64_t sf_cols)
{
    NVQ_CHECK_ARG(x && codes && sf && tscale, NVQ_ERR_ARG, "%s: null pointer argument", fn);
    NVQ_CHECK_ARG(rows >= 1 && rows <= (1ll << 24), NVQ_ERR_SHAPE, "%s: rows outside [1, 2^24]", fn);
    NVQ_CHECK_ARG(K >= 16 && K <= 8192 && K % 16 == 0, NVQ_ERR_SHAPE, "%s: K must be a multiple of 16 in [16, 8192]", fn);
    NVQ_CHECK_ARG(k >= 0 && k <= K && k % 16 == 0, NVQ_ERR_SHAPE, "%s: k=%d must be a multiple of 16 in [0, K]", fn, k);
    NVQ_CHECK_ARG(groups >= 1 && groups <= 4096, NVQ_ERR_SHAPE, "%s: groups outside [1, 4096]", fn);
    NVQ_CHECK_ARG(grp_off || groups == 1 || rows % groups == 0, NVQ_ERR_SHAPE, "%s: rows not divisible by groups", fn);
    NVQ_CHECK_ARG(ldx >= K && ldx % 8 == 0, NVQ_ERR_ALIGN, "%s: ldx must be >= K and a multiple of 8", fn);
    NVQ_CHECK_ARG(ld_codes >= (K + k) / 2 && ld_codes % 16 == 0, NVQ_ERR_ALIGN,
                  "%s: ld_codes must be >= (K+k)/2 and a multiple of 16", fn);
    NVQ_CHECK_ARG(sf_cols >= (K + k) / 16 && sf_cols % 4 == 0, NVQ_ERR_SHAPE,
                  "%s: sf_cols must be >= (K+k)/16 and a multiple of 4", fn);
    NVQ_CHECK_ARG(aligned(codes, 16), NVQ_ERR_ALIGN, "%s: codes must be 16-byte aligned", fn);
    return NVQ_OK;
}

static nvq_status launch_topk(const uint64_t* scores, int64_t K, int32_t groups, int32_t k, int32_t* idx, cudaStream_t st)
{
    topk_kernel<<<groups, kTopkThreads, 0, st>>>(reinterpret_cast<const unsigned long long*>(scores), (int)K, k, idx);
    NVQ_LAUNCH_CHECK("topk_kernel");
    return NVQ_OK;
}

static nvq_status launch_act_tail(const void* x, int64_t rows, int64_t K, int64_t ldx, Groups gr,
                                  const nvq_tensor_scale* tscale, const int32_t* idx, int32_t k, uint8_t* codes,
                                  int64_t ld_codes, uint8_t* sf, int64_t sf_cols, cudaStream_t st)
{
    if (k > 0 && use_row_tail((int)K, k, false) && aligned(x, 16))
        return launch_row_tail<true>(x, ldx, codes, ld_codes, sf, sf_cols, (int)K, k, gr, tscale, idx, 1, st);
    const int64_t tiles = (rows + kTailRows - 1) / kTailRows;
    // split a row's tail blocks over threads until there are ~8 CTAs' worth of threads per SM
    int sms = 148, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    int bsplit = 1;
    const int nbt = k > 0 ? k / 16 : 1;
    while (bsplit < nbt && bsplit < 8 && tiles * bsplit < (int64_t)sms * 8) bsplit *= 2;
    if (bsplit > nbt) bsplit = nbt;
    DeviceStatus* dst = device_status_ptr();
    NVQ_CHECK_ARG(dst, NVQ_ERR_CUDA, "act tail: device status word unavailable");
    act_tail_kernel<<<(unsigned)tiles, kTailRows * bsplit, 0, st>>>(static_cast<const __nv_bfloat16*>(x), ldx, (int)K,
                                                                   k, gr, tscale, idx, codes, ld_codes, sf, sf_cols, bsplit,
                                                                   dst);
    NVQ_LAUNCH_CHECK("act_tail_kernel");
    return NVQ_OK;
}

extern "C" nvq_status rac_select_quantize(const void* x, int64_t rows, int64_t K, int64_t ldx, const int64_t* grp_off,
                                          const int64_t* grp_rows, int32_t groups, const nvq_tensor_scale* tscale,
                                          const uint64_t* scores, int32_t k, uint8_t* codes, int64_t ld_codes,
                                          uint8_t* sf, int64_t sf_cols, int32_t* idx, void* stream)
{
    NVQ_TRACE("rac_select_quantize");
    nvq_status s = check_rac_args("rac_select_quantize", x, rows, K, ldx, grp_off, groups, tscale, k, codes, ld_codes, sf, sf_cols);
    if (s != NVQ_OK) return s;
    NVQ_CHECK_ARG(k == 0 || (scores && idx), NVQ_ERR_ARG, "rac_select_quantize: scores and idx are required when k > 0");
    set_error("");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (k > 0 && (s = launch_topk(scores, K, groups, k, idx, st)) != NVQ_OK) return s;
    return launch_act_tail(x, rows, K, ldx, Groups{grp_off, grp_rows, groups, rows}, tscale, idx, k, codes, ld_codes, sf,
                           sf_cols, st);
}

extern "C" nvq_status rac_select(const uint64_t* scores, int64_t K, int32_t groups, int32_t k, int32_t* idx, void* stream)
{
    NVQ_TRACE("rac_select");
    NVQ_CHECK_ARG(scores && idx, NVQ_ERR_ARG, "rac_select: null pointer argument");
    NVQ_CHECK_ARG(K >= 16 && K <= 8192 && K % 16 == 0, NVQ_ERR_SHAPE, "rac_select: K must be a multiple of 16 in [16, 8192]");
    NVQ_CHECK_ARG(k >= 16 && k <= K && k % 16 == 0, NVQ_ERR_SHAPE, "rac_select: k=%d must be a multiple of 16 in [16, K]", k);
    NVQ_CHECK_ARG(groups >= 1 && groups <= 4096, NVQ_ERR_SHAPE, "rac_select: groups outside [1, 4096]");
    set_error("");
    return launch_topk(scores, K, groups, k, idx, static_cast<cudaStream_t>(stream));
}

extern "C" nvq_status rac_residual_tail(const void* x, int64_t rows, int64_t K, int64_t ldx, const int64_t* grp_off,
                                        const int64_t* grp_rows, int32_t groups, const nvq_tensor_scale* tscale,
                                        const int32_t* idx, int32_t k, uint8_t* codes, int64_t ld_codes, uint8_t* sf,
                                        int64_t sf_cols, void* stream)
{
    NVQ_TRACE("rac_residual_tail");
    nvq_status s = check_rac_args("rac_residual_tail", x, rows, K, ldx, grp_off, groups, tscale, k, codes, ld_codes, sf, sf_cols);
    if (s != NVQ_OK) return s;
    NVQ_CHECK_ARG(k == 0 || idx, NVQ_ERR_ARG, "rac_residual_tail: idx is required when k > 0");
    set_error("");
    return launch_act_tail(x, rows, K, ldx, Groups{grp_off, grp_rows, groups, rows}, tscale, idx, k, codes, ld_codes, sf,
                           sf_cols, static_cast<cudaStream_t>(stream));
}

extern "C" nvq_status nvfp4_channel_major(int32_t groups, int64_t N, int64_t K, const uint8_t* b_codes, int64_t ldb,
                                          const uint8_t* b_sf, int64_t b_sf_cols, uint8_t* cm_codes, uint8_t* cm_sf,
                                          void* stream)
{
    NVQ_TRACE("nvfp4_channel_major");
    NVQ_CHECK_ARG(b_codes && b_sf && cm_codes && cm_sf, NVQ_ERR_ARG, "nvfp4_channel_major: null pointer argument");
    NVQ_CHECK_ARG(groups >= 1 && groups <= 4096 && N >= 64 && N % 64 == 0 && (int64_t)groups * N <= (1ll << 24),
                  NVQ_ERR_SHAPE, "nvfp4_channel_major: N must be a positive multiple of 64 and groups*N <= 2^24");
    NVQ_CHECK_ARG(K >= 16 && K <= 8192 && K % 16 == 0, NVQ_ERR_SHAPE, "nvfp4_channel_major: K must be a multiple of 16 in [16, 8192]");
    NVQ_CHECK_ARG(ldb % 16 == 0 && ldb >= K / 2 && aligned(b_codes, 16) && aligned(cm_codes, 16), NVQ_ERR_ALIGN,
                  "nvfp4_channel_major: b_codes and cm_codes must be 16-byte aligned, ldb a multiple of 16");
    NVQ_CHECK_ARG(b_sf_cols % 4 == 0 && b_sf_cols >= K / 16, NVQ_ERR_SHAPE, "nvfp4_channel_major: b_sf_cols too small");
    set_error("");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const dim3 grid((unsigned)((K + 127) / 128), (unsigned)(N / 64), (unsigned)groups);
    channel_major_codes_kernel<<<grid, 256, 0, st>>>(b_codes, ldb, N, (int)K, cm_codes);
    NVQ_LAUNCH_CHECK("channel_major_codes_kernel");
    const int64_t total = (int64_t)groups * (K / 16) * N;
    channel_major_sf_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(b_sf, b_sf_cols, N, (int)(K / 16), groups, cm_sf);
    NVQ_LAUNCH_CHECK("channel_major_sf_kernel");
    return NVQ_OK;
}

extern "C" nvq_status rac_weight_tail(int32_t groups, int64_t N, int64_t K, int32_t k, const int32_t* idx,
                                      int32_t idx_per_group, uint8_t* b_codes, int64_t ldb, uint8_t* b_sf,
                                      int64_t b_sf_cols, const nvq_tensor_scale* b_tscale, const uint8_t* cm_codes,
                                      const uint8_t* cm_sf, void* stream)
{
    NVQ_TRACE("rac_weight_tail");
    NVQ_CHECK_ARG(idx && b_codes && b_sf && b_tscale, NVQ_ERR_ARG, "rac_weight_tail: null pointer argument");
    NVQ_CHECK_ARG(!cm_codes == !cm_sf, NVQ_ERR_ARG, "rac_weight_tail: give both channel-major arrays or neither");
    NVQ_CHECK_ARG(!cm_codes || N % 64 == 0, NVQ_ERR_SHAPE, "rac_weight_tail: the channel-major path needs N % 64 == 0");
    NVQ_CHECK_ARG(!cm_codes || (aligned(cm_codes, 16) && aligned(cm_sf, 16)), NVQ_ERR_ALIGN,
                  "rac_weight_tail: the channel-major arrays must be 16-byte aligned");
    NVQ_CHECK_ARG(groups >= 1 && groups <= 4096 && N >= 1 && (int64_t)groups * N <= (1ll << 24), NVQ_ERR_SHAPE,
                  "rac_weight_tail: groups*N outside [1, 2^24]");
    NVQ_CHECK_ARG(K >= 16 && K <= 8192 && K % 16 == 0, NVQ_ERR_SHAPE, "rac_weight_tail: K must be a multiple of 16 in [16, 8192]");
    NVQ_CHECK_ARG(k >= 16 && k <= K && k % 16 == 0, NVQ_ERR_SHAPE, "rac_weight_tail: k=%d must be a multiple of 16 in [16, K]", k);
    NVQ_CHECK_ARG(ldb % 16 == 0 && ldb >= (K + k) / 2 && aligned(b_codes, 16), NVQ_ERR_ALIGN,
                  "rac_weight_tail: ldb must be a multiple of 16 covering (K+k)/2 bytes");
    NVQ_CHECK_ARG(b_sf_cols % 4 == 0 && b_sf_cols >= (K + k) / 16, NVQ_ERR_SHAPE, "rac_weight_tail: b_sf_cols too small");
    set_error("");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (use_row_tail((int)K, k, cm_codes != nullptr))
        return launch_row_tail<false>(nullptr, 0, b_codes, ldb, b_sf, b_sf_cols, (int)K, k,
                                      Groups{nullptr, nullptr, groups, (int64_t)groups * N}, b_tscale, idx, idx_per_group, st);
    if (!cm_codes) return weight_tail_impl(b_codes, ldb, b_sf, b_sf_cols, N, (int)K, k, groups, b_tscale, idx, idx_per_group, st);
    const size_t smem = (size_t)(k < kWtChunk ? k : kWtChunk) * 96;
    const dim3 grid((unsigned)(N / kWtRows), (unsigned)groups, (unsigned)((k + kWtChunk - 1) / kWtChunk));
    const int split = k / 16 < kWtMaxSplit ? k / 16 : kWtMaxSplit;  // threads per row
    DeviceStatus* dst = device_status_ptr();
    NVQ_CHECK_ARG(dst, NVQ_ERR_CUDA, "rac_weight_tail: device status word unavailable");
    weight_tail_cm_kernel<<<grid, kWtRows * split, smem, st>>>(b_codes, ldb, b_sf, b_sf_cols, N, (int)K, k, b_tscale, idx,
                                                      idx_per_group, cm_codes, cm_sf, dst);
    NVQ_LAUNCH_CHECK("weight_tail_cm_kernel");
    return NVQ_OK;
}
