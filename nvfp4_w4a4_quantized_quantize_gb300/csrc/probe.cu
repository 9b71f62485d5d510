// probe.cu -- measured NVFP4 tensor-core rate of this GPU: a loop of
// tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X (M128 N256 K64) with no
// memory traffic, one CTA per SM, optionally with three scale-factor copies into TMEM per MMA.
// The result is a roofline reference for the block-scaled GEMM.  The copy variant is a separate
// instantiation: measured on GB300, a loop that merely contains a (never taken) branch around
// tcgen05.cp issues the MMAs at 185 cycles each instead of 128.
#include <cuda.h>

#include "common.cuh"

namespace nvq {

namespace {

constexpr int kProbeThreads = 128;
constexpr uint32_t kIdescProbe = (1u << 7) | (1u << 10) | ((uint32_t)(256 >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);

__device__ __forceinline__ uint32_t psmem(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t pdesc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t layout)
{
    return (uint64_t)((addr & 0x3ffffu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3fffu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3fffu) << 32) | (1ull << 46) | ((uint64_t)layout << 61);
}

template <bool kWithCp>
__global__ void __launch_bounds__(kProbeThreads, 1) mma_rate_kernel(int mmas, DeviceStatus* st, unsigned long long limit)
{
    extern __shared__ __align__(1024) uint8_t sm_raw[];
    __shared__ __align__(8) uint64_t done;
    __shared__ uint32_t tslot;
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    // operands: A 128 x 128 B, B 256 x 128 B, scales 3 x 512 B (value 1.0 = 0x38), codes 0x22 (1.0)
    for (int i = threadIdx.x; i < (16384 + 32768) / 4; i += kProbeThreads)
        reinterpret_cast<uint32_t*>(sm)[i] = 0x22222222u;
    for (int i = threadIdx.x; i < 1536 / 4; i += kProbeThreads) reinterpret_cast<uint32_t*>(sm + 49152)[i] = 0x38383838u;
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(psmem(&done)));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(psmem(&tslot)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = tslot;
    if (threadIdx.x == 0) {
        const uint32_t base = psmem(sm);
        const uint64_t ad = pdesc(base, 16, 1024, 2), bd = pdesc(base + 16384, 16, 1024, 2);
        const uint64_t sd0 = pdesc(base + 49152, 0, 128, 0), sd1 = pdesc(base + 49664, 0, 128, 0),
                       sd2 = pdesc(base + 50176, 0, 128, 0);
        const uint32_t sfa = tmem + 256, sfb = tmem + 260;
        asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(sfa), "l"(sd0) : "memory");
        asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(sfb), "l"(sd1) : "memory");
        asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(sfb + 4), "l"(sd2) : "memory");
        for (int i = 0; i < mmas; ++i) {
            if (kWithCp) {
                asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(sfa), "l"(sd0) : "memory");
                asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(sfb), "l"(sd1) : "memory");
                asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(sfb + 4), "l"(sd2) : "memory");
            }
            asm volatile(
                "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(
                    tmem),
                "l"(ad + 2 * (i & 3)), "l"(bd + 2 * (i & 3)), "r"(kIdescProbe), "r"(i > 0 ? 1u : 0u), "r"(sfa), "r"(sfb)
                : "memory");
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(psmem(&done))
                     : "memory");
        // bounded wait for the MMAs to finish
        const long long t0 = clock64();
        uint32_t ok = 0;
        while (!ok) {
            asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                         : "=r"(ok)
                         : "r"(psmem(&done))
                         : "memory");
            if (!ok && (unsigned long long)(clock64() - t0) > limit) {
                report_timeout(st, 31);
                break;
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
}

}  // namespace

}  // namespace nvq

using namespace nvq;

/* Measured rate of back-to-back M128 N256 K64 NVFP4 MMAs on every SM (FP32 accumulation in
 * TMEM, no memory traffic); with_cp adds the three scale-factor copies per MMA that the GEMM
 * issues.  Synchronous: returns the achieved TFLOP/s in *tflops. */
extern "C" nvq_status nvq_fp4_mma_rate(int32_t mmas_per_sm, int32_t with_cp, float* tflops, void* stream)
{
    NVQ_TRACE("nvq_fp4_mma_rate");
    NVQ_CHECK_ARG(tflops && mmas_per_sm >= 16 && mmas_per_sm <= (1 << 20), NVQ_ERR_ARG, "nvq_fp4_mma_rate: bad arguments");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    DeviceStatus* ds = device_status_ptr();
    NVQ_CHECK_ARG(ds, NVQ_ERR_CUDA, "nvq_fp4_mma_rate: device status word unavailable");
    const int smem = 50688 + 1024;
    auto kernel = with_cp ? mma_rate_kernel<true> : mma_rate_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return cuda_status(e, "cudaFuncSetAttribute(mma_rate_kernel)");
    // warm-up, then the timed launch
    kernel<<<sms, kProbeThreads, smem, st>>>(64, ds, wait_limit());
    cudaEvent_t a, b;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    cudaEventRecord(a, st);
    kernel<<<sms, kProbeThreads, smem, st>>>(mmas_per_sm, ds, wait_limit());
    cudaEventRecord(b, st);
    e = cudaEventSynchronize(b);
    float ms = 0.0f;
    cudaEventElapsedTime(&ms, a, b);
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    if (e != cudaSuccess) return cuda_status(e, "mma_rate_kernel");
    *tflops = (float)(2.0 * 128 * 256 * 64 * (double)mmas_per_sm * sms / (ms * 1e-3) / 1e12);
    set_error("");
    return NVQ_OK;
}
