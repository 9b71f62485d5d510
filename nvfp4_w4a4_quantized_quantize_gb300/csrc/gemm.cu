// gemm.cu -- native block-scaled NVFP4 W4A4 grouped GEMM with the RAC correction carried as
// extra K-columns (QUADS §3.3 "Targeted residual compensation": the correction runs on the
// same W4A4 FP4 tensor-core path; §4.4.2: FP4 tensor-core kernels are the throughput point).
//
// Y[r, n] = alpha_g * sum_{c < K+k} V[a_rc] sa_{r,c/16} V[b_nc] sb_{n,c/16},
// alpha_g = S_dec(A_g) * S_dec(W_g), for the rows r of group g and the weight rows of group g.
//
// sm_103a design (one CTA per SM, persistent):
//   tile 128 x 256 x 256 (M x N x K-tile of FP4 elements = 128 bytes per row) per CTA; tiles run
//   N-fastest inside each 128-row block, so the CTAs working at the same time read one A block
//   and one group's weights, which L2 serves to all of them;
//   warps 0, 14, 15  TMA producers (A; the two 128-row halves of B, or all of B and the B
//              scales): code tiles by cp.async.bulk.tensor (128-byte swizzle, out-of-range
//              columns zero-filled), scale atoms by cp.async.bulk (the blocked scale layout
//              makes every 128-row x 64-column scale tile one contiguous 512 B); three issuing
//              warps fill shared memory faster than one;
//   warp 1     TMEM allocator and MMA issuer: per K-tile, once the stage's scales are in
//              TMEM, tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X (K = 64 each, UE4M3
//              scales, FP32 accumulation in TMEM), tcgen05.commit to free the stage;
//   warps 2-5  scale staging, one warp per TMEM lane quarter: the stage's scale atoms from
//              shared memory into registers and into TMEM with tcgen05.st (the layout the
//              block-scaled MMA reads: every lane quarter holds each atom's 32 x 16 bytes).
//              Register stores keep the scales off the tensor pipe's copy path, which at
//              12 small copies per K-tile cost about 40% of the MMA rate;
//   warps 6-13 epilogue: tcgen05.ld of the accumulator, alpha scaling, bf16 store, with the
//              SwiGLU or routing-weight variants; the routing-weight tile goes out through a
//              swizzled shared-memory buffer per warp as TMA tile stores.
// The same kernel, instantiated for E4M3 operands (kind::mxf8f6f4, scale_vec::1X, one UE8M0
// scale per 32 elements, K = 32 per MMA, 128 elements per 128-byte K-tile row, no tensor
// scale), is the FP8 W8A8 block-scaled baseline the paper compares against (§2.2 "FP8",
// §4.4.2): a stage then holds one scale atom per 128 rows, and MMA j of the stage reads byte j
// of each scale word (the scale-factor ID fields of the instruction descriptor).
// Every mbarrier wait is bounded; on expiry the kernel records NVQ_ERR_TIMEOUT and unwinds.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cstring>

#include "common.cuh"

namespace nvq {

constexpr int kBM = 128, kBN = 256;
constexpr int kRowBytes = 128;              // bytes of a K-tile row in shared memory = swizzle span
// Epilogue staging for the coalesced bf16 stores (one 32-row x 128-byte buffer per epilogue warp).
constexpr int kStagingBytes = 8 * 32 * 128;
constexpr int kStagesMax = 4;               // 4 x 54 KB for FP4 (a 128-element K-tile in 8 x 27 KB was
                                            // slower: twice the per-stage hand-offs)
constexpr uint32_t kSwizzleLayout = 2u;     // tcgen05 smem layout: 128-byte swizzle
constexpr uint32_t kSBO = 8 * kRowBytes;    // stride between 8-row core-matrix groups
constexpr int kABytes = kBM * kRowBytes;    // 16384
constexpr int kBBytes = kBN * kRowBytes;    // 32768
constexpr int kMmaPerStage = 4;             // 32 bytes of every tile row per MMA
constexpr int kThreads = 512;  // warps 0, 14, 15 TMA, warp 1 MMA, warps 2-5 scale staging, warps 6-13 epilogue
constexpr int kFirstEpiWarp = 6;
constexpr int kProducers = 3;       // one TMA box per stage each: A, weight rows half 0, half 1
constexpr int kProdWarpB0 = 14, kProdWarpB1 = 15;
constexpr int kEpiThreads = 256;
constexpr int kMaxGroups = 512;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 0;                  // 256 fp32 columns
constexpr uint32_t kSFCol = 256;                 // + stage * F::kSFColsPerStage

// Operand formats.  A scale atom is the blocked layout's 512 bytes: 128 rows x 4 scale columns.
struct Fp4 {  // NVFP4: E2M1 x E2M1, one UE4M3 scale per 16 elements, scale_vec::4X
    static constexpr int kElemsPerStage = 256;  // per 128-byte row
    static constexpr int kMmaK = 64;
    static constexpr int kSfVec = 16;
    // A/B format E2M1 (1) in bits 7-9 / 10-12, K-major A and B, N >> 3 in bits 17-22, scale
    // type UE4M3 (bit 23 = 0), M >> 4 in bits 24-28.
    static constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
    static constexpr uint32_t idesc(int) { return kIdesc; }
    __device__ static void mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t sfa_tmem,
                               uint32_t sfb_tmem, uint32_t accumulate)
    {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
                d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
            : "memory");
    }
};

struct Fp8 {  // FP8: E4M3 x E4M3, one UE8M0 scale per 32 elements, scale_vec::1X
    static constexpr int kElemsPerStage = 128;
    static constexpr int kMmaK = 32;
    static constexpr int kSfVec = 32;
    // A/B format E4M3 (0), K-major, N >> 3 in bits 17-22, scale type UE8M0 (bit 23 = 1),
    // M >> 4 in bits 24-28; the scale-factor IDs (byte of the 32-bit scale word) of B in bits
    // 4-5 and of A in bits 29-30.
    static constexpr uint32_t kIdesc = ((uint32_t)(kBN >> 3) << 17) | (1u << 23) | ((uint32_t)(kBM >> 4) << 24);
    static constexpr uint32_t idesc(int j) { return kIdesc | ((uint32_t)j << 4) | ((uint32_t)j << 29); }
    __device__ static void mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t sfa_tmem,
                               uint32_t sfb_tmem, uint32_t accumulate)
    {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
                d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
            : "memory");
    }
};

// Per-format stage geometry.
template <class F>
struct Geo {
    static constexpr int kSfAtoms = F::kElemsPerStage / (4 * F::kSfVec);  // per 128 rows: FP4 4, FP8 1
    static constexpr int kSFABytes = 512 * kSfAtoms;
    static constexpr int kSFBBytes = 1024 * kSfAtoms;                     // 2 row blocks
    static constexpr int kStageBytes = (kABytes + kBBytes + kSFABytes + kSFBBytes + 1023) / 1024 * 1024;
    static constexpr int kSmemBytes(int stages, bool staged) { return stages * kStageBytes + (staged ? kStagingBytes : 0) + 1024; }
    static constexpr uint32_t kSFColsPerStage = 12 * kSfAtoms;            // SFA 4 + SFB 8 per atom
    // scale atom of MMA j of a stage (FP4: one per MMA; FP8: one for all four)
    static constexpr int atom_of(int j) { return (j * F::kMmaK) / (4 * F::kSfVec); }
    // atoms holding the scales of the first n MMAs
    static constexpr int atoms_for(int n_mma) { return (n_mma * F::kMmaK + 4 * F::kSfVec - 1) / (4 * F::kSfVec); }
};
static_assert(Geo<Fp4>::kStageBytes == 55296 && Geo<Fp8>::kStageBytes == 51200, "stage sizes");

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
    nvq_tensor_scale* out_ts;  // NULL, or per-group max |out| (bf16 epilogues) into .amax
    int32_t out_tma;           // staged epilogue: full 32-row pieces leave by TMA store (tmap_out)
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
                                          int where, bool draining = false)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (!draining && *abort_flag) return false;
        if ((unsigned long long)(clock64() - t0) > (draining ? drain_limit(a.wait_limit) : a.wait_limit)) {
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

// Two 32-column accumulator loads, one wait.
__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, uint32_t tb, float* va, float* vb)
{
    uint32_t r[64];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
          "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
          "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
          "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
          "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(ta), "r"(tb)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        va[i] = __uint_as_float(r[i]);
        vb[i] = __uint_as_float(r[32 + i]);
    }
}

// Six 16-column accumulator loads (addresses t[0..5]), one wait: 96 values.
__device__ __forceinline__ void tmem_ld16x6(const uint32_t* t, float* v)
{
    uint32_t r[96];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%96];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%97];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47}, [%98];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%99];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79}, [%100];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95}, [%101];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95])
        : "r"(t[0]), "r"(t[1]), "r"(t[2]), "r"(t[3]), "r"(t[4]), "r"(t[5])
        : "memory");
#pragma unroll
    for (int i = 0; i < 96; ++i) v[i] = __uint_as_float(r[i]);
}

// Two 16-column accumulator loads, one wait: 32 values.
__device__ __forceinline__ void tmem_ld16x2(uint32_t ta, uint32_t tb, float* v)
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(ta), "r"(tb)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// 4 / 8 / 16 / 32 consecutive TMEM columns of this warp's 32 lanes from registers.
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t* v)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]),
                 "r"(v[3])
                 : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* v)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
                 "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* v)
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
        "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]),
        "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
        "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

// n32 consecutive 32-byte pieces of packed words to global memory: 256-bit stores when the
// destination is 32-byte aligned (wide), 128-bit stores otherwise.
template <int kWords>
__device__ __forceinline__ void store_row(void* dst, const uint32_t* w, bool wide)
{
    if (wide) {
#pragma unroll
        for (int i = 0; i < kWords / 8; ++i)
            asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(reinterpret_cast<uint32_t*>(dst) + 8 * i),
                         "r"(w[8 * i]), "r"(w[8 * i + 1]), "r"(w[8 * i + 2]), "r"(w[8 * i + 3]), "r"(w[8 * i + 4]),
                         "r"(w[8 * i + 5]), "r"(w[8 * i + 6]), "r"(w[8 * i + 7])
                         : "memory");
    } else {
        uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int i = 0; i < kWords / 4; ++i) d[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    }
}

// max |bf16| over n packed bf16x2 words (exact: a maximum of bf16 values).
template <int kWords>
__device__ __forceinline__ float amax_packed(const uint32_t* w)
{
    uint32_t m = 0;
#pragma unroll
    for (int i = 0; i < kWords; ++i) {
        // sign-cleared bf16 values order like their bit patterns: an integer max per half
        const uint32_t v = w[i] & 0x7fff7fffu;
        m = __vmaxu2(m, v);
    }
    const uint32_t hi = m >> 16, lo = m & 0xffffu;
    return __uint_as_float((hi > lo ? hi : lo) << 16);
}

// Warp maximum of a non-negative value, folded into *dst (float bits ordered as integers).
__device__ __forceinline__ void warp_amax_to(float v, float* dst)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((threadIdx.x & 31) == 0 && v > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(dst), __float_as_uint(v));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// 2^x and 1/x on the special-function unit (approximate; |x| large gives inf / 0 as IEEE).
__device__ __forceinline__ float ex2_approx(float x)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ float rcp_approx(float x)
{
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// ------------------------------------------------------------------ tile scheduling
struct Tile {
    int g;
    int row0;       // first A row of this CTA's 128-row tile (rows < 2^24)
    int rows;       // valid rows in the tile (1..128)
    int nt;         // N tile
};

// Per-group tables in shared memory, filled once per CTA: first row, row count and the prefix
// of 128-row tiles.  Tiles run N-fastest inside each 128-row block, so that the CTAs working at
// the same time share one A block (read from HBM once) and one group's weights (kept in L2).
struct GroupTab {
    int start[kMaxGroups];
    int rows[kMaxGroups];
    int mt_pre[kMaxGroups + 1];
};

__device__ __forceinline__ Tile tile_of(int64_t t, int n_tiles, const GroupTab& tab, int G)
{
    Tile T;
    T.nt = (int)(t % n_tiles);
    const int gm = (int)(t / n_tiles);  // global 128-row tile index
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tab.mt_pre[mid] <= gm) lo = mid; else hi = mid - 1;
    }
    T.g = lo;
    const int mt = gm - tab.mt_pre[lo];
    T.row0 = tab.start[lo] + mt * kBM;
    const int left = tab.rows[lo] - mt * kBM;
    T.rows = left < kBM ? left : kBM;
    return T;
}

// ------------------------------------------------------------------ the kernel
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                                 uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Shared memory -> global tile store (bulk async group of the issuing thread).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(smem_u32(src))
                 : "memory");
}

// One 64-column piece of an epilogue warp's 32 rows (pk: this thread's row, 32 words = 64 bf16)
// through the warp's 4 KB shared-memory buffer: 16-byte units XOR-swizzled by row (the 128-byte
// swizzle of a TMA box, conflict-free both ways).  A piece of 32 rows inside the tile leaves as
// one TMA tile store (32 x 64 bf16); a ragged piece leaves as whole 128-byte row pieces, four
// rows per store instruction, up to the last row (rvalid).
__device__ __forceinline__ void staged_piece(const CUtensorMap* tmap_out, __nv_bfloat16* out, int64_t ldo, uint8_t* buf,
                                             const uint32_t* pk, int64_t rbase, int rvalid, int64_t col, bool by_tma)
{
    const int lane = threadIdx.x & 31;
    if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");  // the buffer has been read out
    __syncwarp();
#pragma unroll
    for (int u = 0; u < 8; ++u)
        *reinterpret_cast<uint4*>(buf + lane * 128 + ((u ^ (lane & 7)) << 4)) =
            make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
    if (by_tma) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the TMA unit
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmap_out, buf, (int)col, (int)rbase);
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
    } else {
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int r = 4 * j + (lane >> 3), u = lane & 7;
            const uint4 d = *reinterpret_cast<const uint4*>(buf + r * 128 + ((u ^ (r & 7)) << 4));
            if (r < rvalid) *reinterpret_cast<uint4*>(out + (rbase + r) * ldo + col + 8 * u) = d;
        }
    }
}

// kStages: depth of the operand ring; kStaged: the bf16 store and routing-weight epilogues write
// through a per-warp shared-memory buffer and TMA stores (needs the room of one stage: the ring
// is 3 deep then).
template <class F, int kStages, bool kStaged>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                                                           const __grid_constant__ CUtensorMap tmap_b,
                                                           const __grid_constant__ CUtensorMap tmap_b256,
                                                           const __grid_constant__ CUtensorMap tmap_out, const GemmArgs a)
{
    using GF = Geo<F>;
    constexpr int kStageBytes = GF::kStageBytes;
    constexpr int kSfAtoms = GF::kSfAtoms;
    constexpr int kSFABytes = GF::kSFABytes, kSFBBytes = GF::kSFBBytes;
    constexpr uint32_t kSFColsPerStage = GF::kSFColsPerStage;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kStages], sf_bar[kStages], empty_bar[kStages], acc_full, acc_empty, drain_bar;
    __shared__ uint32_t tmem_base_slot;
    __shared__ GroupTab tab;
    __shared__ int abort_flag;

    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.gr.G;

    // per-group tables: rows and starts in parallel, the tile prefix by warp 0
    for (int g = threadIdx.x; g < G; g += kThreads) {
        int64_t gb, ge;
        group_range(a.gr, g, gb, ge);
        tab.start[g] = (int)gb;
        tab.rows[g] = ge > gb ? (int)(ge - gb) : 0;
    }
    if (threadIdx.x == 0) {
        abort_flag = 0;
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full_bar[i], kProducers);  // each producer's box
            mbar_init(&sf_bar[i], 4);  // the four scale-staging warps
            mbar_init(&empty_bar[i], 1);  // the MMA commit releases a stage
        }
        mbar_init(&acc_full, 1);
        mbar_init(&acc_empty, kEpiThreads);
        mbar_init(&drain_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");  // visible to the async proxy
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    if (warp == 0) {
        constexpr int kPer = kMaxGroups / 32;
        int cnt[kPer], sum = 0;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int g = lane * kPer + i;
            cnt[i] = g < G ? (tab.rows[g] + kBM - 1) / kBM : 0;
            sum += cnt[i];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        int run = incl - sum;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int g = lane * kPer + i;
            if (g <= G) tab.mt_pre[g] = run;
            run += cnt[i];
        }
        if (lane == 31 && G == kMaxGroups) tab.mt_pre[G] = run;
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
    const int total_mtiles = tab.mt_pre[G];
    const int n_tiles = (int)(a.N / kBN);
    const int64_t total_tiles = (int64_t)total_mtiles * n_tiles;
    const int num_kt = (a.ktot + F::kElemsPerStage - 1) / F::kElemsPerStage;
    volatile int* abrt = &abort_flag;

    const int prod = warp == 0 ? 0 : (warp == kProdWarpB0 ? 1 : (warp == kProdWarpB1 ? 2 : -1));
    if (prod >= 0) {
        // ---------------- producers: the TMA engine sustains more per SM with fewer, larger
        // requests and with requests from several warps, so each stage is loaded by three:
        // warp 0 the A tile and its scale atoms; when the weight tile's 256 rows are contiguous
        // (every epilogue but SwiGLU) warp 14 loads them as one box and warp 15 their scale
        // atoms, otherwise warps 14 and 15 one 128-row half each with its scale atoms.  Weight
        // loads are L2 evict-last: every 128-row block of the group re-reads them.
        uint64_t pol_keep;
        asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol_keep));
        int stage = 0;
        uint32_t phase = 0, issued = 0;
        for (int64_t t = blockIdx.x; t < total_tiles && !*abrt; t += gridDim.x) {
            const Tile T = tile_of(t, n_tiles, tab, G);
            int64_t brow;
            if (a.epilogue == NVQ_EPI_SWIGLU)
                brow = (int64_t)T.g * a.N + (int64_t)T.nt * (kBN / 2) + (prod == 2 ? a.N / 2 : 0);
            else
                brow = (int64_t)T.g * a.N + (int64_t)T.nt * kBN + (prod == 2 ? kBN / 2 : 0);
            if (lane == 0) {
                for (int kt = 0; kt < num_kt; ++kt) {
                    if (!mbar_wait(&empty_bar[stage], phase ^ 1, a, abrt, 1)) break;
                    const int kleft = a.ktot - kt * F::kElemsPerStage;
                    const int n_mma = kleft >= F::kElemsPerStage ? kMmaPerStage : (kleft + F::kMmaK - 1) / F::kMmaK;
                    const uint32_t sf_bytes = 512u * GF::atoms_for(n_mma);
                    uint8_t* sA = smem + stage * kStageBytes;
                    if (prod == 0) {
                        mbar_expect_tx(&full_bar[stage], kABytes + sf_bytes);
                        tma_load_2d(sA, &tmap_a, kt * kRowBytes, T.row0, &full_bar[stage]);
                        bulk_load(sA + kABytes + kBBytes,
                                  a.a_sf + ((int64_t)(T.row0 >> 7) * (a.a_sf_cols >> 2) + kt * kSfAtoms) * 512, sf_bytes,
                                  &full_bar[stage]);
                    } else if (a.epilogue == NVQ_EPI_SWIGLU) {
                        const int h = prod - 1;
                        mbar_expect_tx(&full_bar[stage], kBBytes / 2 + sf_bytes);
                        tma_load_2d_hint(sA + kABytes + h * (kBBytes / 2), &tmap_b, kt * kRowBytes, (int)brow, &full_bar[stage],
                                         pol_keep);
                        bulk_load(sA + kABytes + kBBytes + kSFABytes + h * (kSFBBytes / 2),
                                  a.b_sf + ((brow >> 7) * (a.b_sf_cols >> 2) + kt * kSfAtoms) * 512, sf_bytes, &full_bar[stage]);
                    } else if (prod == 1) {  // brow: the tile's first weight row
                        mbar_expect_tx(&full_bar[stage], kBBytes);
                        tma_load_2d_hint(sA + kABytes, &tmap_b256, kt * kRowBytes, (int)brow, &full_bar[stage], pol_keep);
                    } else {  // brow: the tile's second 128-row block
                        mbar_expect_tx(&full_bar[stage], 2 * sf_bytes);
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            bulk_load(sA + kABytes + kBBytes + kSFABytes + h * (kSFBBytes / 2),
                                      a.b_sf + (((brow >> 7) - 1 + h) * (a.b_sf_cols >> 2) + kt * kSfAtoms) * 512, sf_bytes,
                                      &full_bar[stage]);
                    }
                    ++issued;
                    if (++stage == kStages) { stage = 0; phase ^= 1; }
                }
            }
            __syncwarp();
        }
        if (*abrt && lane == 0) {
            // let this producer's copies still in flight land before the CTA can exit: its last
            // issue on each stage is the phase (phase ^ 1) for stages before `stage`, else `phase`
            // (a phase another producer left incomplete only makes this wait use its bound)
            for (int s = 0; s < kStages; ++s)
                if (issued > (uint32_t)s) mbar_wait(&full_bar[s], s < stage ? phase : phase ^ 1, a, abrt, 11, true);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer: waits for the stage's scale factors to be in TMEM (which
        // implies its operand tiles are in shared memory), then up to 4 MMAs and one commit
        // that frees the stage.  Descriptors are precomputed; nothing else is in this loop.
        // MMA j reads scale atom atom_of(j) (SFA 4 columns, SFB 8 columns per atom) and, for
        // FP8, byte j of its scale words.
        const uint32_t base = smem_u32(smem);
        const uint64_t a_desc0 = smem_desc(base, 16, kSBO, kSwizzleLayout);
        const uint64_t b_desc0 = smem_desc(base + kABytes, 16, kSBO, kSwizzleLayout);
        constexpr uint64_t kStageStep = kStageBytes >> 4;
        int stage = 0;
        uint32_t phase = 0, acc_phase = 0;
        bool issued_any = false;
        for (int64_t t = blockIdx.x; t < total_tiles && !*abrt; t += gridDim.x) {
            if (!mbar_wait(&acc_empty, acc_phase ^ 1, a, abrt, 2)) break;
            tc_fence_after();
            bool ok = true;
            for (int kt = 0; kt < num_kt; ++kt) {
                if (!mbar_wait(&sf_bar[stage], phase, a, abrt, 3)) { ok = false; break; }
                tc_fence_after();
                const int kleft = a.ktot - kt * F::kElemsPerStage;
                const int n_mma = kleft >= F::kElemsPerStage ? kMmaPerStage : (kleft + F::kMmaK - 1) / F::kMmaK;
                if (lane == 0) {
                    const uint64_t so = (uint64_t)stage * kStageStep;
                    const uint32_t sfa_t = tmem + kSFCol + stage * kSFColsPerStage;
                    const uint32_t sfb_t = sfa_t + 4 * kSfAtoms;
#pragma unroll
                    for (int j = 0; j < kMmaPerStage; ++j)  // step j: 32 bytes into the tile rows
                        if (j < n_mma)
                            F::mma(tmem + kAccCol, a_desc0 + so + 2 * j, b_desc0 + so + 2 * j, F::idesc(j),
                                   sfa_t + 4 * GF::atom_of(j), sfb_t + 8 * GF::atom_of(j), (kt > 0 || j > 0) ? 1u : 0u);
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
            mbar_wait(&drain_bar, 0, a, abrt, 12, true);
        }
        __syncwarp();
    } else if (warp < kFirstEpiWarp) {
        // ---------------- scale staging (warps 2-5, TMEM lane quarter = warp % 4): per K-tile,
        // lane i loads row i (16 bytes) of each of the stage's 3 * kSfAtoms scale atoms from
        // shared memory and stores them to its TMEM lane, SFA atom j at columns 4j, SFB atom j
        // of weight half h at 4 kSfAtoms + 8j + 4h; then fence and arrive on sf_bar for the MMA
        // warp.
        const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
        int stage = 0;
        uint32_t phase = 0;
        for (int64_t t = blockIdx.x; t < total_tiles && !*abrt; t += gridDim.x) {
            bool ok = true;
            for (int kt = 0; kt < num_kt; ++kt) {
                if (!mbar_wait(&full_bar[stage], phase, a, abrt, 5)) { ok = false; break; }
                const uint8_t* sf = smem + stage * kStageBytes + kABytes + kBBytes + lane * 16;
                uint32_t va[4 * kSfAtoms], vb[8 * kSfAtoms];
#pragma unroll
                for (int j = 0; j < kSfAtoms; ++j) {
                    const uint4 x = *reinterpret_cast<const uint4*>(sf + j * 512);
                    va[4 * j] = x.x; va[4 * j + 1] = x.y; va[4 * j + 2] = x.z; va[4 * j + 3] = x.w;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint4 y = *reinterpret_cast<const uint4*>(sf + kSFABytes + h * (kSFBBytes / 2) + j * 512);
                        vb[8 * j + 4 * h] = y.x; vb[8 * j + 4 * h + 1] = y.y; vb[8 * j + 4 * h + 2] = y.z; vb[8 * j + 4 * h + 3] = y.w;
                    }
                }
                const uint32_t sfa_t = tmem + kSFCol + stage * kSFColsPerStage + lane_addr;
                if constexpr (kSfAtoms == 4) {
                    tmem_st16(sfa_t, va);
                    tmem_st32(sfa_t + 16, vb);
                } else if constexpr (kSfAtoms == 2) {
                    tmem_st8(sfa_t, va);
                    tmem_st16(sfa_t + 8, vb);
                } else {
                    static_assert(kSfAtoms == 1, "scale atoms per stage");
                    tmem_st4(sfa_t, va);
                    tmem_st8(sfa_t + 4, vb);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sf_bar[stage]);
                if (++stage == kStages) { stage = 0; phase ^= 1; }
            }
            if (!ok) break;
        }
    } else {
        // ---------------- epilogue: warps 6..13; TMEM lane quarter = warp % 4, column half =
        // (warp - 6) / 4.  The accumulator is read in 32-column pieces, packed to bf16 as it
        // comes, and released once the last piece is in registers; the last piece's arithmetic
        // and the global stores overlap the next tile's MMAs.
        const int quarter = warp & 3;
        const int half = (warp - kFirstEpiWarp) >> 2;
        const int r_in_tile = quarter * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const bool wide = (a.ldo % 16) == 0 && (reinterpret_cast<uintptr_t>(a.out) % 32) == 0;
        uint32_t acc_phase = 0;
        for (int64_t t = blockIdx.x; t < total_tiles && !*abrt; t += gridDim.x) {
            const Tile T = tile_of(t, n_tiles, tab, G);
            const bool valid = r_in_tile < T.rows;
            const int64_t grow = (int64_t)T.row0 + r_in_tile;
            // NVFP4: alpha_g = S_dec(A) S_dec(W); FP8 (no tensor scales): 1
            const float alpha = a.a_ts ? __fmul_rn(a.a_ts[a.a_ts_per_group ? T.g : 0].s_dec, a.b_ts[T.g].s_dec) : 1.0f;
            const float w = (a.epilogue == NVQ_EPI_ROW_SCALE && valid) ? a.row_w[grow] : 1.0f;
            if (!mbar_wait(&acc_full, acc_phase, a, abrt, 4)) break;
            tc_fence_after();
            const uint32_t tacc = tmem + kAccCol + lane_addr;
            // the staged instantiation runs only the routing-weight epilogue (launch_gemm): the
            // fp32 and SwiGLU branches are compiled out of it, which keeps its registers
            if (!kStaged && a.epilogue == NVQ_EPI_STORE_F32) {
                float* orow = reinterpret_cast<float*>(a.out) + grow * a.ldo + (int64_t)T.nt * kBN + half * (kBN / 2);
#pragma unroll 1
                for (int c = 0; c < kBN / 2; c += 64) {
                    float v0[32], v1[32];
                    tmem_ld32x2(tacc + half * (kBN / 2) + c, tacc + half * (kBN / 2) + c + 32, v0, v1);
                    if (valid) {
                        float4* d = reinterpret_cast<float4*>(orow + c);
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            d[i] = make_float4(__fmul_rn(alpha, v0[4 * i]), __fmul_rn(alpha, v0[4 * i + 1]),
                                               __fmul_rn(alpha, v0[4 * i + 2]), __fmul_rn(alpha, v0[4 * i + 3]));
                            d[8 + i] = make_float4(__fmul_rn(alpha, v1[4 * i]), __fmul_rn(alpha, v1[4 * i + 1]),
                                                   __fmul_rn(alpha, v1[4 * i + 2]), __fmul_rn(alpha, v1[4 * i + 3]));
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(&acc_empty);
            } else if (!kStaged && a.epilogue == NVQ_EPI_SWIGLU) {
                // gate columns [half*64, +64), up columns [128 + half*64, +64) -> h columns [half*64, +64)
                const uint64_t alpha2 = f2pack(alpha, alpha);
                const uint64_t nlog2e2 = f2pack(-1.4426950408889634f, -1.4426950408889634f);  // -log2(e)
                const uint64_t one2 = f2pack(1.0f, 1.0f);
                // the accumulator in 16-column pieces (gate and up halves of each): three pieces
                // are read before any arithmetic, the first one's SwiGLU runs, the last piece is
                // read and the accumulator released, so only a quarter of the arithmetic comes
                // before the release
                // silu(g) u = g u / (1 + 2^(-g log2 e)), element pairs on the paired fp32
                // instructions (the epilogue is bound by instruction issue at two warps per
                // scheduler), the power of two and the reciprocal on the special-function unit
                uint32_t pk[32];
                auto swiglu8 = [&](const float* g, const float* u, uint32_t* out) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint64_t gp = f2mul(alpha2, f2pack(g[2 * i], g[2 * i + 1]));
                        const uint64_t up = f2mul(alpha2, f2pack(u[2 * i], u[2 * i + 1]));
                        float t0, t1;
                        f2unpack(f2mul(gp, nlog2e2), t0, t1);
                        float d0, d1;
                        f2unpack(f2add(f2pack(ex2_approx(t0), ex2_approx(t1)), one2), d0, d1);
                        float h0, h1;
                        f2unpack(f2mul(f2mul(gp, f2pack(rcp_approx(d0), rcp_approx(d1))), up), h0, h1);
                        out[i] = pack_bf16x2(h0, h1);
                    }
                };
                {
                    float v[96];  // pieces 0..2: gate 16, up 16 each
                    const uint32_t tg = tacc + half * 64, tu = tacc + kBN / 2 + half * 64;
                    const uint32_t t6[6] = {tg, tu, tg + 16, tu + 16, tg + 32, tu + 32};
                    tmem_ld16x6(t6, v);
                    swiglu8(v, v + 16, pk);
                    float w[32];  // piece 3
                    tmem_ld16x2(tg + 48, tu + 48, w);
                    tc_fence_before();
                    mbar_arrive(&acc_empty);  // released: the rest overlaps the next tile's MMAs
                    swiglu8(v + 32, v + 48, pk + 8);
                    swiglu8(v + 64, v + 80, pk + 16);
                    swiglu8(w, w + 16, pk + 24);
                }
                if (valid) store_row<32>(a.out + grow * a.ldo + (int64_t)T.nt * (kBN / 2) + half * 64, pk, wide);
                if (a.out_ts) warp_amax_to(valid ? amax_packed<32>(pk) : 0.0f, &a.out_ts[T.g].amax);
            } else {
                const float sc = (a.epilogue == NVQ_EPI_ROW_SCALE) ? w : 1.0f;
                const uint64_t alpha2 = f2pack(alpha, alpha), sc2 = f2pack(sc, sc);
                uint32_t pk[64];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    float v0[32], v1[32];
                    tmem_ld32x2(tacc + half * (kBN / 2) + 64 * c, tacc + half * (kBN / 2) + 64 * c + 32, v0, v1);
                    if (c == 1) {  // released once the last piece is in registers
                        tc_fence_before();
                        mbar_arrive(&acc_empty);
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) {  // fl(fl(alpha acc) w), element pairs per instruction
                        uint64_t yp = f2mul(alpha2, f2pack(v0[2 * i], v0[2 * i + 1]));
                        uint64_t zp = f2mul(alpha2, f2pack(v1[2 * i], v1[2 * i + 1]));
                        if (a.epilogue == NVQ_EPI_ROW_SCALE) {
                            yp = f2mul(yp, sc2);
                            zp = f2mul(zp, sc2);
                        }
                        float y0, y1, z0, z1;
                        f2unpack(yp, y0, y1);
                        f2unpack(zp, z0, z1);
                        pk[32 * c + i] = pack_bf16x2(y0, y1);
                        pk[32 * c + 16 + i] = pack_bf16x2(z0, z1);
                    }
                }
                if constexpr (kStaged) {
                    const int rvalid = T.rows - quarter * 32;  // rows of this warp's 32 inside the tile
#pragma unroll
                    for (int c = 0; c < 2; ++c)
                        staged_piece(&tmap_out, a.out, a.ldo, smem + kStages * kStageBytes + (warp - kFirstEpiWarp) * 4096,
                                     pk + 32 * c, (int64_t)T.row0 + quarter * 32, rvalid,
                                     (int64_t)T.nt * kBN + half * (kBN / 2) + 64 * c, a.out_tma && rvalid >= 32);
                } else if (valid) {
                    store_row<64>(a.out + grow * a.ldo + (int64_t)T.nt * kBN + half * (kBN / 2), pk, wide);
                }
                if (a.out_ts) warp_amax_to(valid ? amax_packed<64>(pk) : 0.0f, &a.out_ts[T.g].amax);
            }
            acc_phase ^= 1;
        }
        // the TMA stores this thread issued have finished (reading shared memory and writing)
        if (kStaged && lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
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

// 2D byte tensor map over FP4 codes, swizzled as the K-tile's row width (kRowBytes); box =
// kRowBytes x box_rows rows.
static nvq_status make_map(CUtensorMap* m, const void* base, int64_t inner_bytes, int64_t rows, int64_t ld,
                           uint32_t box_rows = 128)
{
    auto enc = get_encode();
    NVQ_CHECK_ARG(enc, NVQ_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[2] = {(cuuint64_t)inner_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld};
    cuuint32_t box[2] = {(cuuint32_t)kRowBytes, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, kRowBytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    NVQ_CHECK_ARG(r == CUDA_SUCCESS, NVQ_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return NVQ_OK;
}

// 2D bf16 tensor map over the output rows for the staged epilogue's TMA stores: box 64 columns
// (128 bytes, 128-byte swizzle, as the staging buffer is laid out) x 32 rows.
static nvq_status make_out_map(CUtensorMap* m, const void* out, int64_t width, int64_t rows, int64_t ldo)
{
    auto enc = get_encode();
    NVQ_CHECK_ARG(enc, NVQ_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ldo * 2)};
    cuuint32_t box[2] = {64, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(out), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    NVQ_CHECK_ARG(r == CUDA_SUCCESS, NVQ_ERR_CUDA, "cuTensorMapEncodeTiled (output) failed (%d)", (int)r);
    return NVQ_OK;
}

nvq_status weight_tail_impl(uint8_t* codes, int64_t ld_codes, uint8_t* sf, int64_t sf_cols, int64_t N, int K, int k,
                            int G, const nvq_tensor_scale* ts, const int32_t* idx, int idx_per_group, cudaStream_t st);

// Persistent launch: one CTA per SM, no more CTAs than tiles.
template <class F, int kStages, bool kStaged>
nvq_status launch_gemm_cfg(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mb256, const CUtensorMap& mo,
                           const GemmArgs& ga, int32_t groups, int64_t N, cudaStream_t st)
{
    constexpr int kSmem = Geo<F>::kSmemBytes(kStages, kStaged);
    static_assert(kSmem + 8 * 1024 <= 227 * 1024, "shared memory of the GEMM");
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel<F, kStages, kStaged>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return cuda_status(e, "cudaFuncSetAttribute(gemm_kernel)");
    // an upper bound of the tiles: every group adds at most one partial 128-row tile
    const int64_t max_tiles = (int64_t)(ga.total_mtiles_max + groups) * (N / kBN);
    const int ctas = (int)(max_tiles < sms ? max_tiles : sms);
    gemm_kernel<F, kStages, kStaged><<<ctas, kThreads, kSmem, st>>>(ma, mb, mb256, mo, ga);
    NVQ_LAUNCH_CHECK("gemm_kernel");
    return NVQ_OK;
}

// The routing-weight epilogue (the down projection: a full 128 x 256 bf16 tile per output,
// written to memory once and read back by the combine) stores through shared memory, by TMA,
// with a 3-deep operand ring; the other epilogues keep the 4-deep ring and plain stores (their
// longer K loops lose more to the shallower ring than their stores gain: gate/up 0.2925 ->
// 0.2945 ms, dense 0.1287 -> 0.1314 ms at the prefill and 4096 x 14336 x 4160 shapes).
template <class F>
nvq_status launch_gemm(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mb256, GemmArgs ga, int32_t groups,
                       int64_t N, cudaStream_t st)
{
    CUtensorMap mo;
    memset(&mo, 0, sizeof(mo));
    ga.out_tma = 0;
    if (ga.epilogue == NVQ_EPI_ROW_SCALE) {
        nvq_status s = make_out_map(&mo, ga.out, N, ga.gr.total_rows, ga.ldo);
        if (s != NVQ_OK) return s;
        ga.out_tma = 1;
        return launch_gemm_cfg<F, 3, true>(ma, mb, mb256, mo, ga, groups, N, st);
    }
    return launch_gemm_cfg<F, kStagesMax, false>(ma, mb, mb256, mo, ga, groups, N, st);
}

// Arguments shared by both entries.
static nvq_status check_gemm_common(const char* fn, int32_t groups, const int64_t* grp_off, int64_t rows, int64_t N,
                                    int32_t epilogue, const float* row_w, int64_t ldo, const void* out)
{
    NVQ_CHECK_ARG(epilogue == NVQ_EPI_STORE || epilogue == NVQ_EPI_SWIGLU || epilogue == NVQ_EPI_ROW_SCALE ||
                      epilogue == NVQ_EPI_STORE_F32, NVQ_ERR_ARG, "%s: unknown epilogue %d", fn, epilogue);
    NVQ_CHECK_ARG(epilogue != NVQ_EPI_ROW_SCALE || row_w, NVQ_ERR_ARG, "%s: row_w required", fn);
    NVQ_CHECK_ARG(groups >= 1 && groups <= kMaxGroups, NVQ_ERR_SHAPE, "%s: groups outside [1, %d]", fn, kMaxGroups);
    NVQ_CHECK_ARG(grp_off || groups == 1, NVQ_ERR_SHAPE, "%s: grp_off required when groups > 1", fn);
    NVQ_CHECK_ARG(rows >= 1 && rows <= (1ll << 24), NVQ_ERR_SHAPE, "%s: rows outside [1, 2^24]", fn);
    NVQ_CHECK_ARG(N >= kBN && N % kBN == 0 && (int64_t)groups * N <= (1ll << 24), NVQ_ERR_SHAPE,
                  "%s: N=%lld must be a positive multiple of %d", fn, (long long)N, kBN);
    NVQ_CHECK_ARG(ldo % 8 == 0 && ldo >= (epilogue == NVQ_EPI_SWIGLU ? N / 2 : N), NVQ_ERR_ALIGN,
                  "%s: ldo must be a multiple of 8 covering the output width", fn);
    NVQ_CHECK_ARG(aligned(out, 16), NVQ_ERR_ALIGN, "%s: out must be 16-byte aligned", fn);
    return NVQ_OK;
}

static GemmArgs gemm_args(int32_t groups, const int64_t* grp_off, const int64_t* grp_rows, int64_t rows,
                          const uint8_t* a_sf, int64_t a_sf_cols, const uint8_t* b_sf, int64_t b_sf_cols, int64_t N,
                          int64_t ktot, int32_t epilogue, const float* row_w, void* out, int64_t ldo)
{
    GemmArgs ga;
    ga.gr = Groups{grp_off, grp_rows, groups, rows};
    ga.total_mtiles_max = (int)((rows + kBM - 1) / kBM);
    ga.a_sf = a_sf;
    ga.a_sf_cols = a_sf_cols;
    ga.b_sf = b_sf;
    ga.b_sf_cols = b_sf_cols;
    ga.a_ts = nullptr;
    ga.a_ts_per_group = 0;
    ga.b_ts = nullptr;
    ga.N = N;
    ga.ktot = (int32_t)ktot;
    ga.epilogue = epilogue;
    ga.row_w = row_w;
    ga.out = static_cast<__nv_bfloat16*>(out);  // fp32 rows for NVQ_EPI_STORE_F32
    ga.ldo = ldo;
    ga.status = device_status_ptr();
    ga.wait_limit = wait_limit();
    ga.out_ts = nullptr;
    ga.out_tma = 0;
    return ga;
}

}  // namespace nvq

using namespace nvq;

extern "C" nvq_status w4a4_rac_grouped_gemm(int32_t groups, const int64_t* grp_off, const int64_t* grp_rows, int64_t rows,
                                            const uint8_t* a_codes, int64_t lda, const uint8_t* a_sf, int64_t a_sf_cols,
                                            const nvq_tensor_scale* a_tscale, int32_t a_scale_per_group,
                                            uint8_t* b_codes, int64_t ldb, uint8_t* b_sf, int64_t b_sf_cols,
                                            const nvq_tensor_scale* b_tscale, int64_t N, int64_t K, int32_t k,
                                            const int32_t* idx, int32_t idx_per_group, int32_t epilogue,
                                            const float* row_w, void* out, int64_t ldo, nvq_tensor_scale* out_tscale,
                                            void* stream)
{
    NVQ_TRACE("w4a4_rac_grouped_gemm");
    static const char* fn = "w4a4_rac_grouped_gemm";
    NVQ_CHECK_ARG(a_codes && a_sf && a_tscale && b_codes && b_sf && b_tscale && out, NVQ_ERR_ARG, "%s: null pointer argument", fn);
    nvq_status s = check_gemm_common(fn, groups, grp_off, rows, N, epilogue, row_w, ldo, out);
    if (s != NVQ_OK) return s;
    NVQ_CHECK_ARG(K >= 16 && K <= 8192 && K % 16 == 0, NVQ_ERR_SHAPE, "%s: K must be a multiple of 16 in [16, 8192]", fn);
    NVQ_CHECK_ARG(k >= 0 && k <= K && k % 16 == 0, NVQ_ERR_SHAPE, "%s: k=%d must be a multiple of 16 in [0, K]", fn, k);
    const int64_t ktot = K + k;
    NVQ_CHECK_ARG(lda % 16 == 0 && ldb % 16 == 0 && lda >= ktot / 2 && ldb >= ktot / 2, NVQ_ERR_ALIGN,
                  "%s: lda/ldb must be multiples of 16 covering (K+k)/2 bytes", fn);
    NVQ_CHECK_ARG(a_sf_cols % 4 == 0 && b_sf_cols % 4 == 0 && a_sf_cols >= nvq_sf_cols(ktot) && b_sf_cols >= nvq_sf_cols(ktot),
                  NVQ_ERR_SHAPE, "%s: sf_cols must be >= nvq_sf_cols(K+k)", fn);
    NVQ_CHECK_ARG(aligned(a_codes, 16) && aligned(b_codes, 16) && aligned(a_sf, 16) && aligned(b_sf, 16), NVQ_ERR_ALIGN,
                  "%s: operands must be 16-byte aligned", fn);
    NVQ_CHECK_ARG(!out_tscale || epilogue != NVQ_EPI_STORE_F32, NVQ_ERR_ARG, "%s: out_tscale needs a bf16 epilogue", fn);
    set_error("");
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    if (idx && k > 0) {
        s = weight_tail_impl(b_codes, ldb, b_sf, b_sf_cols, N, (int)K, k, groups, b_tscale, idx, idx_per_group, st);
        if (s != NVQ_OK) return s;
    }

    CUtensorMap ma, mb, mb256;
    s = make_map(&ma, a_codes, ktot / 2, rows, lda);
    if (s != NVQ_OK) return s;
    s = make_map(&mb, b_codes, ktot / 2, (int64_t)groups * N, ldb);
    if (s != NVQ_OK) return s;
    s = make_map(&mb256, b_codes, ktot / 2, (int64_t)groups * N, ldb, 256);
    if (s != NVQ_OK) return s;

    GemmArgs ga = gemm_args(groups, grp_off, grp_rows, rows, a_sf, a_sf_cols, b_sf, b_sf_cols, N, ktot, epilogue, row_w,
                            out, ldo);
    ga.a_ts = a_tscale;
    ga.a_ts_per_group = a_scale_per_group;
    ga.b_ts = b_tscale;
    ga.out_ts = out_tscale;
    NVQ_CHECK_ARG(ga.status, NVQ_ERR_CUDA, "%s: device status word unavailable", fn);
    if (out_tscale) {
        const cudaError_t me = cudaMemsetAsync(out_tscale, 0, sizeof(nvq_tensor_scale) * groups, st);
        if (me != cudaSuccess) return cuda_status(me, "cudaMemsetAsync(out_tscale)");
    }
    return launch_gemm<Fp4>(ma, mb, mb256, ga, groups, N, st);
}

extern "C" nvq_status fp8_blockscaled_grouped_gemm(int32_t groups, const int64_t* grp_off, const int64_t* grp_rows,
                                                   int64_t rows, const uint8_t* a_codes, int64_t lda, const uint8_t* a_sf,
                                                   int64_t a_sf_cols, const uint8_t* b_codes, int64_t ldb,
                                                   const uint8_t* b_sf, int64_t b_sf_cols, int64_t N, int64_t K,
                                                   int32_t epilogue, const float* row_w, void* out, int64_t ldo,
                                                   void* stream)
{
    NVQ_TRACE("fp8_blockscaled_grouped_gemm");
    static const char* fn = "fp8_blockscaled_grouped_gemm";
    NVQ_CHECK_ARG(a_codes && a_sf && b_codes && b_sf && out, NVQ_ERR_ARG, "%s: null pointer argument", fn);
    nvq_status s = check_gemm_common(fn, groups, grp_off, rows, N, epilogue, row_w, ldo, out);
    if (s != NVQ_OK) return s;
    NVQ_CHECK_ARG(K >= 32 && K <= 16384 && K % 32 == 0, NVQ_ERR_SHAPE, "%s: K must be a multiple of 32 in [32, 16384]", fn);
    NVQ_CHECK_ARG(lda % 16 == 0 && ldb % 16 == 0 && lda >= K && ldb >= K, NVQ_ERR_ALIGN,
                  "%s: lda/ldb must be multiples of 16 covering K bytes", fn);
    NVQ_CHECK_ARG(a_sf_cols % 4 == 0 && b_sf_cols % 4 == 0 && a_sf_cols >= nvq_fp8_sf_cols(K) && b_sf_cols >= nvq_fp8_sf_cols(K),
                  NVQ_ERR_SHAPE, "%s: sf_cols must be >= nvq_fp8_sf_cols(K)", fn);
    NVQ_CHECK_ARG(aligned(a_codes, 16) && aligned(b_codes, 16) && aligned(a_sf, 16) && aligned(b_sf, 16), NVQ_ERR_ALIGN,
                  "%s: operands must be 16-byte aligned", fn);
    set_error("");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    CUtensorMap ma, mb, mb256;
    s = make_map(&ma, a_codes, K, rows, lda);
    if (s != NVQ_OK) return s;
    s = make_map(&mb, b_codes, K, (int64_t)groups * N, ldb);
    if (s != NVQ_OK) return s;
    s = make_map(&mb256, b_codes, K, (int64_t)groups * N, ldb, 256);
    if (s != NVQ_OK) return s;
    GemmArgs ga = gemm_args(groups, grp_off, grp_rows, rows, a_sf, a_sf_cols, b_sf, b_sf_cols, N, K, epilogue, row_w, out, ldo);
    NVQ_CHECK_ARG(ga.status, NVQ_ERR_CUDA, "%s: device status word unavailable", fn);
    return launch_gemm<Fp8>(ma, mb, mb256, ga, groups, N, st);
}
