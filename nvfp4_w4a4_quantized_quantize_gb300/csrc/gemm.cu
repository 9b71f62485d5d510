// gemm.cu -- native block-scaled NVFP4 W4A4 grouped GEMM with the RAC correction carried as
// extra K-columns (QUADS §3.3 "Targeted residual compensation": the correction runs on the
// same W4A4 FP4 tensor-core path; §4.4.2: FP4 tensor-core kernels are the throughput point).
//
// Y[r, n] = alpha_g * sum_{c < K+k} V[a_rc] sa_{r,c/16} V[b_nc] sb_{n,c/16},
// alpha_g = S_dec(A_g) * S_dec(W_g), for the rows r of group g and the weight rows of group g.
//
// sm_103a design (one CTA per SM, persistent):
//   tile 128 x 256 x 256 (M x N x K-tile of FP4 elements = 128 bytes per row);
//   warp 0     TMA producer: A and B code tiles by cp.async.bulk.tensor (128-byte swizzle,
//              out-of-range columns zero-filled), scale atoms by cp.async.bulk (the blocked
//              scale layout makes every 128-row x 64-column scale tile one contiguous 512 B);
//   warp 1     TMEM allocator and MMA issuer: per K-tile, tcgen05.cp of the scale atoms into
//              TMEM, then tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X (K = 64 each,
//              UE4M3 scales, FP32 accumulation in TMEM), tcgen05.commit to free the stage;
//   warps 2-5  epilogue: tcgen05.ld of the accumulator, alpha scaling, bf16 store, with the
//              SwiGLU or routing-weight variants.
// Every mbarrier wait is bounded; on expiry the kernel records NVQ_ERR_TIMEOUT and unwinds.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace nvq {

constexpr int kBM = 128, kBN = 256, kBK = 256;  // kBK in FP4 elements
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK / 2;     // 16384
constexpr int kBBytes = kBN * kBK / 2;     // 32768
constexpr int kSFABytes = kBM * kBK / 16;  // 2048: 4 atoms of 512 B
constexpr int kSFBBytes = kBN * kBK / 16;  // 4096: 2 row blocks x 4 atoms
constexpr int kStageBytes = kABytes + kBBytes + kSFABytes + kSFBBytes;  // 55296 (54 x 1024)
constexpr int kSmemBytes = kStages * kStageBytes + 1024;
constexpr int kThreads = 192;
constexpr int kMaxGroups = 512;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0;                  // 256 fp32 columns
constexpr uint32_t kSFCol = 256;                 // + stage * 48: SFA 16 columns, SFB 32 columns
constexpr uint32_t kSFColsPerStage = 48;

struct GemmArgs {
    Groups gr;              // A row groups
    int32_t total_mtiles_max;
    const uint8_t* a_sf;
    int64_t a_sf_cols;
    const uint8_t* b_sf;
    int64_t b_sf_cols;
    const nvq_tensor_scale* a_ts;
    int32_t a_ts_per_group;
    const nvq_tensor_scale* b_ts;
    int64_t N;              // weight rows per group
    int32_t ktot;           // K + k
    int32_t epilogue;
    const float* row_w;
    __nv_bfloat16* out;
    int64_t ldo;
    DeviceStatus* status;
    unsigned long long wait_limit;
};

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait; returns false (after recording the timeout) if the limit ran out or another
// role of the CTA already gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const GemmArgs& a, volatile int* abort_flag,
                                          int where)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if ((unsigned long long)(clock64() - t0) > a.wait_limit) {
            report_timeout(a.status, where);
            *abort_flag = 1;
            return false;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start >> 4, LBO >> 4, SBO >> 4, version 1,
// layout type in bits 61-63 (0 = no swizzle, 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout)
{
    return (uint64_t)((addr & 0x3ffffu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3fffu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3fffu) << 32) | (1ull << 46) | ((uint64_t)layout << 61);
}

// Instruction descriptor, block-scaled kinds: A/B format E2M1 (1) in bits 7-9 / 10-12,
// K-major A and B, N >> 3 in bits 17-22, scale type UE4M3 (bit 23 = 0), M >> 4 in bits 24-28.
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);

__device__ __forceinline__ void mma_fp4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t sfa_tmem,
                                        uint32_t sfb_tmem, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
            d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(kIdesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

__device__ __forceinline__ void tc_cp_sf(uint32_t tmem, uint64_t sdesc)
{
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(tmem), "l"(sdesc) : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v)
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const float* v)
{
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        pk[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
}

// ------------------------------------------------------------------ tile scheduling
struct Tile {
    int g;
    int64_t row0;   // first A row of the tile
    int rows;       // valid rows in the tile (<= 128)
    int nt;         // N tile
};

__device__ __forceinline__ Tile tile_of(int64_t t, int total_mtiles, const int* mt_pre, const GemmArgs& a)
{
    Tile T;
    T.nt = (int)(t / total_mtiles);
    const int gm = (int)(t % total_mtiles);
    int lo = 0, hi = a.gr.G - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (mt_pre[mid] <= gm) lo = mid; else hi = mid - 1;
    }
    T.g = lo;
    int64_t gb, ge;
    group_range(a.gr, lo, gb, ge);
    const int mt = gm - mt_pre[lo];
    T.row0 = gb + (int64_t)mt * kBM;
    const int64_t left = ge - T.row0;
    T.rows = (int)(left < kBM ? left : kBM);
    return T;
}

// ------------------------------------------------------------------ the kernel
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                                                           const __grid_constant__ CUtensorMap tmap_b, const GemmArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kStages], empty_bar[kStages], acc_full, acc_empty, drain_bar;
    __shared__ uint32_t tmem_base_slot;
    __shared__ int mt_pre[kMaxGroups + 1];
    __shared__ int abort_flag;

    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // group m-tile prefix
    if (threadIdx.x == 0) {
        int s = 0;
        for (int g = 0; g < a.gr.G; ++g) {
            mt_pre[g] = s;
            int64_t gb, ge;
            group_range(a.gr, g, gb, ge);
            const int64_t n = ge > gb ? ge - gb : 0;
            s += (int)((n + kBM - 1) / kBM);
        }
        mt_pre[a.gr.G] = s;
        abort_flag = 0;
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], 1);
        }
        mbar_init(&acc_full, 1);
        mbar_init(&acc_empty, 128);
        mbar_init(&drain_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_slot;
    const int total_mtiles = mt_pre[a.gr.G];
    const int n_tiles = (int)(a.N / kBN);
    const int64_t total_tiles = (int64_t)total_mtiles * n_tiles;
    const int num_kt = (a.ktot + kBK - 1) / kBK;
    volatile int* abrt = &abort_flag;

    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            for (int64_t t = blockIdx.x; t < total_tiles && !*abrt; t += gridDim.x) {
                const Tile T = tile_of(t, total_mtiles, mt_pre, a);
                int64_t brow0, brow1;
                if (a.epilogue == NVQ_EPI_SWIGLU) {
                    brow0 = (int64_t)T.g * a.N + (int64_t)T.nt * (kBN / 2);
                    brow1 = brow0 + a.N / 2;
                } else {
                    brow0 = (int64_t)T.g * a.N + (int64_t)T.nt * kBN;
                    brow1 = brow0 + kBN / 2;
                }
                for (int kt = 0; kt < num_kt; ++kt) {
                    if (!mbar_wait(&empty_bar[stage], phase ^ 1, a, abrt, 1)) break;
                    const int kleft = a.ktot - kt * kBK;
                    const int n_atoms = kleft >= kBK ? 4 : (kleft + 63) / 64;
                    uint8_t* sA = smem + stage * kStageBytes;
                    uint8_t* sB = sA + kABytes;
                    uint8_t* sSFA = sB + kBBytes;
                    uint8_t* sSFB = sSFA + kSFABytes;
                    mbar_expect_tx(&full_bar[stage], kABytes + kBBytes + 3u * 512u * n_atoms);
                    tma_load_2d(sA, &tmap_a, kt * (kBK / 2), (int)T.row0, &full_bar[stage]);
                    tma_load_2d(sB, &tmap_b, kt * (kBK / 2), (int)brow0, &full_bar[stage]);
                    tma_load_2d(sB + kBBytes / 2, &tmap_b, kt * (kBK / 2), (int)brow1, &full_bar[stage]);
                    const uint8_t* srcA = a.a_sf + ((T.row0 >> 7) * (a.a_sf_cols >> 2) + kt * 4) * 512;
                    bulk_load(sSFA, srcA, 512u * n_atoms, &full_bar[stage]);
                    const uint8_t* srcB0 = a.b_sf + ((brow0 >> 7) * (a.b_sf_cols >> 2) + kt * 4) * 512;
                    const uint8_t* srcB1 = a.b_sf + ((brow1 >> 7) * (a.b_sf_cols >> 2) + kt * 4) * 512;
                    bulk_load(sSFB, srcB0, 512u * n_atoms, &full_bar[stage]);
                    bulk_load(sSFB + kSFBBytes / 2, srcB1, 512u * n_atoms, &full_bar[stage]);
                    if (++stage == kStages) { stage = 0; phase ^= 1; }
                }
            }
            if (*abrt) {
                // let issued copies land before the CTA can exit
                for (int s = 0; s < kStages; ++s) mbar_wait(&full_bar[s], 0, a, abrt, 11) || mbar_wait(&full_bar[s], 1, a, abrt, 11);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        int stage = 0;
        uint32_t phase = 0, acc_phase = 0;
        bool issued_any = false;
        for (int64_t t = blockIdx.x; t < total_tiles && !*abrt; t += gridDim.x) {
            if (!mbar_wait(&acc_empty, acc_phase ^ 1, a, abrt, 2)) break;
            tc_fence_after();
            bool ok = true;
            for (int kt = 0; kt < num_kt; ++kt) {
                if (!mbar_wait(&full_bar[stage], phase, a, abrt, 3)) { ok = false; break; }
                tc_fence_after();
                const int kleft = a.ktot - kt * kBK;
                const int n_mma = kleft >= kBK ? 4 : (kleft + 63) / 64;
                if (lane == 0) {
                    uint8_t* sA = smem + stage * kStageBytes;
                    uint8_t* sB = sA + kABytes;
                    uint8_t* sSFA = sB + kBBytes;
                    uint8_t* sSFB = sSFA + kSFABytes;
                    const uint32_t sfa_t = tmem + kSFCol + stage * kSFColsPerStage;
                    const uint32_t sfb_t = sfa_t + 16;
                    for (int j = 0; j < n_mma; ++j) {
                        tc_cp_sf(sfa_t + 4 * j, smem_desc(smem_u32(sSFA + 512 * j), 0, 128, 0));
                        tc_cp_sf(sfb_t + 8 * j, smem_desc(smem_u32(sSFB + 512 * j), 0, 128, 0));
                        tc_cp_sf(sfb_t + 8 * j + 4, smem_desc(smem_u32(sSFB + kSFBBytes / 2 + 512 * j), 0, 128, 0));
                    }
                    for (int j = 0; j < n_mma; ++j) {
                        const uint64_t ad = smem_desc(smem_u32(sA) + 32 * j, 16, 1024, 2);
                        const uint64_t bd = smem_desc(smem_u32(sB) + 32 * j, 16, 1024, 2);
                        mma_fp4(tmem + kAccCol, ad, bd, sfa_t + 4 * j, sfb_t + 8 * j, (kt > 0 || j > 0) ? 1u : 0u);
                    }
                    tc_commit(&empty_bar[stage]);
                    issued_any = true;
                }
                __syncwarp();
                if (++stage == kStages) { stage = 0; phase ^= 1; }
            }
            if (!ok) break;
            if (lane == 0) tc_commit(&acc_full);
            __syncwarp();
            acc_phase ^= 1;
        }
        if (*abrt && issued_any && lane == 0) {
            tc_commit(&drain_bar);
            mbar_wait(&drain_bar, 0, a, abrt, 12);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue (warps 2..5 -> TMEM lane quarters 2, 3, 0, 1)
        const int quarter = warp & 3;
        const int r_in_tile = quarter * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        uint32_t acc_phase = 0;
        for (int64_t t = blockIdx.x; t < total_tiles && !*abrt; t += gridDim.x) {
            const Tile T = tile_of(t, total_mtiles, mt_pre, a);
            if (!mbar_wait(&acc_full, acc_phase, a, abrt, 4)) break;
            tc_fence_after();
            const float alpha =
                __fmul_rn(a.a_ts[a.a_ts_per_group ? T.g : 0].s_dec, a.b_ts[T.g].s_dec);
            const bool valid = r_in_tile < T.rows;
            const int64_t grow = T.row0 + r_in_tile;
            float v[32], u[32];
            if (a.epilogue == NVQ_EPI_SWIGLU) {
                __nv_bfloat16* orow = a.out + grow * a.ldo + (int64_t)T.nt * (kBN / 2);
#pragma unroll 1
                for (int c = 0; c < kBN / 2; c += 32) {
                    tmem_ld32(tmem + kAccCol + lane_addr + c, v);
                    tmem_ld32(tmem + kAccCol + lane_addr + kBN / 2 + c, u);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float g = __fmul_rn(alpha, v[i]);
                        const float up = __fmul_rn(alpha, u[i]);
                        v[i] = __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), up);
                    }
                    if (valid) store_bf16x32(orow + c, v);
                }
            } else if (a.epilogue == NVQ_EPI_STORE_F32) {
                float* orow = reinterpret_cast<float*>(a.out) + grow * a.ldo + (int64_t)T.nt * kBN;
#pragma unroll 1
                for (int c = 0; c < kBN; c += 32) {
                    tmem_ld32(tmem + kAccCol + lane_addr + c, v);
                    if (valid) {
                        float4* d = reinterpret_cast<float4*>(orow + c);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            d[i] = make_float4(__fmul_rn(alpha, v[4 * i]), __fmul_rn(alpha, v[4 * i + 1]),
                                               __fmul_rn(alpha, v[4 * i + 2]), __fmul_rn(alpha, v[4 * i + 3]));
                    }
                }
            } else {
                const float w = (a.epilogue == NVQ_EPI_ROW_SCALE && valid) ? a.row_w[grow] : 1.0f;
                __nv_bfloat16* orow = a.out + grow * a.ldo + (int64_t)T.nt * kBN;
#pragma unroll 1
                for (int c = 0; c < kBN; c += 32) {
                    tmem_ld32(tmem + kAccCol + lane_addr + c, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        v[i] = __fmul_rn(alpha, v[i]);
                        if (a.epilogue == NVQ_EPI_ROW_SCALE) v[i] = __fmul_rn(v[i], w);
                    }
                    if (valid) store_bf16x32(orow + c, v);
                }
            }
            tc_fence_before();
            mbar_arrive(&acc_empty);
            acc_phase ^= 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

// ------------------------------------------------------------------ host side
static PFN_cuTensorMapEncodeTiled_v12000 get_encode()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

static nvq_status make_map(CUtensorMap* m, const void* base, int64_t inner_bytes, int64_t rows, int64_t ld)
{
    auto enc = get_encode();
    NVQ_CHECK_ARG(enc, NVQ_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[2] = {(cuuint64_t)inner_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld};
    cuuint32_t box[2] = {128, 128};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    NVQ_CHECK_ARG(r == CUDA_SUCCESS, NVQ_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return NVQ_OK;
}

nvq_status weight_tail_impl(uint8_t* codes, int64_t ld_codes, uint8_t* sf, int64_t sf_cols, int64_t N, int K, int k,
                            int G, const nvq_tensor_scale* ts, const int32_t* idx, int idx_per_group, cudaStream_t st);

}  // namespace nvq

using namespace nvq;

extern "C" nvq_status w4a4_rac_grouped_gemm(int32_t groups, const int64_t* grp_off, const int64_t* grp_rows, int64_t rows,
                                            const uint8_t* a_codes, int64_t lda, const uint8_t* a_sf, int64_t a_sf_cols,
                                            const nvq_tensor_scale* a_tscale, int32_t a_scale_per_group,
                                            uint8_t* b_codes, int64_t ldb, uint8_t* b_sf, int64_t b_sf_cols,
                                            const nvq_tensor_scale* b_tscale, int64_t N, int64_t K, int32_t k,
                                            const int32_t* idx, int32_t idx_per_group, int32_t epilogue,
                                            const float* row_w, void* out, int64_t ldo, void* stream)
{
    NVQ_CHECK_ARG(a_codes && a_sf && a_tscale && b_codes && b_sf && b_tscale && out, NVQ_ERR_ARG,
                  "w4a4_rac_grouped_gemm: null pointer argument");
    NVQ_CHECK_ARG(epilogue == NVQ_EPI_STORE || epilogue == NVQ_EPI_SWIGLU || epilogue == NVQ_EPI_ROW_SCALE ||
                      epilogue == NVQ_EPI_STORE_F32, NVQ_ERR_ARG,
                  "w4a4_rac_grouped_gemm: unknown epilogue %d", epilogue);
    NVQ_CHECK_ARG(epilogue != NVQ_EPI_ROW_SCALE || row_w, NVQ_ERR_ARG, "w4a4_rac_grouped_gemm: row_w required");
    NVQ_CHECK_ARG(groups >= 1 && groups <= kMaxGroups, NVQ_ERR_SHAPE, "w4a4_rac_grouped_gemm: groups outside [1, %d]", kMaxGroups);
    NVQ_CHECK_ARG(grp_off || groups == 1, NVQ_ERR_SHAPE, "w4a4_rac_grouped_gemm: grp_off required when groups > 1");
    NVQ_CHECK_ARG(rows >= 1 && rows <= (1ll << 24), NVQ_ERR_SHAPE, "w4a4_rac_grouped_gemm: rows outside [1, 2^24]");
    NVQ_CHECK_ARG(N >= kBN && N % kBN == 0 && (int64_t)groups * N <= (1ll << 24), NVQ_ERR_SHAPE,
                  "w4a4_rac_grouped_gemm: N=%lld must be a positive multiple of %d", (long long)N, kBN);
    NVQ_CHECK_ARG(K >= 16 && K <= 8192 && K % 16 == 0, NVQ_ERR_SHAPE, "w4a4_rac_grouped_gemm: K must be a multiple of 16 in [16, 8192]");
    NVQ_CHECK_ARG(k >= 0 && k <= K && k % 16 == 0 && k <= 512, NVQ_ERR_SHAPE, "w4a4_rac_grouped_gemm: bad k=%d", k);
    const int64_t ktot = K + k;
    NVQ_CHECK_ARG(lda % 16 == 0 && ldb % 16 == 0 && lda >= ktot / 2 && ldb >= ktot / 2, NVQ_ERR_ALIGN,
                  "w4a4_rac_grouped_gemm: lda/ldb must be multiples of 16 covering (K+k)/2 bytes");
    NVQ_CHECK_ARG(a_sf_cols % 4 == 0 && b_sf_cols % 4 == 0 && a_sf_cols >= nvq_sf_cols(ktot) && b_sf_cols >= nvq_sf_cols(ktot),
                  NVQ_ERR_SHAPE, "w4a4_rac_grouped_gemm: sf_cols must be >= nvq_sf_cols(K+k)");
    NVQ_CHECK_ARG(ldo % 8 == 0 && ldo >= (epilogue == NVQ_EPI_SWIGLU ? N / 2 : N), NVQ_ERR_ALIGN,
                  "w4a4_rac_grouped_gemm: ldo must be a multiple of 8 covering the output width");
    NVQ_CHECK_ARG(aligned(a_codes, 16) && aligned(b_codes, 16) && aligned(a_sf, 16) && aligned(b_sf, 16) && aligned(out, 16),
                  NVQ_ERR_ALIGN, "w4a4_rac_grouped_gemm: operands must be 16-byte aligned");
    set_error("");
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    nvq_status s = NVQ_OK;
    if (idx && k > 0) {
        s = weight_tail_impl(b_codes, ldb, b_sf, b_sf_cols, N, (int)K, k, groups, b_tscale, idx, idx_per_group, st);
        if (s != NVQ_OK) return s;
    }

    CUtensorMap ma, mb;
    s = make_map(&ma, a_codes, ktot / 2, rows, lda);
    if (s != NVQ_OK) return s;
    s = make_map(&mb, b_codes, ktot / 2, (int64_t)groups * N, ldb);
    if (s != NVQ_OK) return s;

    GemmArgs ga;
    ga.gr = Groups{grp_off, grp_rows, groups, rows};
    ga.total_mtiles_max = (int)((rows + kBM - 1) / kBM);
    ga.a_sf = a_sf;
    ga.a_sf_cols = a_sf_cols;
    ga.b_sf = b_sf;
    ga.b_sf_cols = b_sf_cols;
    ga.a_ts = a_tscale;
    ga.a_ts_per_group = a_scale_per_group;
    ga.b_ts = b_tscale;
    ga.N = N;
    ga.ktot = (int32_t)ktot;
    ga.epilogue = epilogue;
    ga.row_w = row_w;
    ga.out = static_cast<__nv_bfloat16*>(out);  // fp32 rows for NVQ_EPI_STORE_F32
    ga.ldo = ldo;
    ga.status = device_status_ptr();
    ga.wait_limit = wait_limit();
    NVQ_CHECK_ARG(ga.status, NVQ_ERR_CUDA, "w4a4_rac_grouped_gemm: device status word unavailable");

    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t max_tiles = (int64_t)(ga.total_mtiles_max + groups) * (N / kBN);
    const int grid = (int)(max_tiles < sms ? max_tiles : sms);
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return cuda_status(e, "cudaFuncSetAttribute(gemm_kernel)");
    gemm_kernel<<<grid, kThreads, kSmemBytes, st>>>(ma, mb, ga);
    NVQ_LAUNCH_CHECK("gemm_kernel");
    return NVQ_OK;
}
