// A stand-in for the GEMM2 that produces expert_out, for measuring and
// testing the dependent-launch overlap of the finalize.
//
// "FlashInfer MoE 성능 최적화: CuTe DSL을 활용한 Deterministic Finalize
// 개선기" (flashinfer PR 5319 analysis), section 2: the FC2 grouped GEMM
// signals its dependents right after its own input wait, so the standalone
// finalizer can load its independent state while FC2 still runs; the
// finalizer's dependency wait still protects every FC2 output load.  This
// kernel reproduces exactly that protocol around a plain copy: wait, signal,
// optionally busy for a fixed number of cycles (the GEMM's main loop), then
// write the rows.  It is not part of the finalize.
#include <cstdint>

#include <cuda_runtime.h>

#include "moe_finalize_rmsnorm.h"
#include "mfr_device.cuh"
#include "mfr_internal.h"

namespace {

__global__ void __launch_bounds__(256) producer_kernel(const uint4* src, uint4* dst, int64_t n,
                                                       long long busy_cycles) {
    mfr::pdl_wait();                 // the previous kernel may still read dst
    mfr::pdl_launch_dependents();    // the finalize may start its prologue
    if (busy_cycles > 0) {
        const long long t0 = clock64();
        while (clock64() - t0 < busy_cycles) {
        }
    }
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
        dst[i] = src[i];
}

}  // namespace

extern "C" int moe_finalize_rmsnorm_bench_producer(const void* src, void* expert_out, int64_t rows, int64_t H,
                                                   long long busy_cycles, int enable_pdl, void* stream) {
    if (rows < 0 || H < 8 || H % 8 != 0 || busy_cycles < 0 || busy_cycles > 4000000000LL)
        return MFR_ERR_INVALID_ARG;
    if (rows == 0) return MFR_OK;
    if (!src || !expert_out || (reinterpret_cast<uintptr_t>(src) & 15) || (reinterpret_cast<uintptr_t>(expert_out) & 15))
        return MFR_ERR_MISALIGNED;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return MFR_ERR_CUDA;
    }
    const int64_t n = rows * H / 8;
    const int64_t want = (n + 255) / 256;
    const int blocks = static_cast<int>(want < 4LL * sms ? want : 4LL * sms);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    if (enable_pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    if (cudaLaunchKernelEx(&cfg, producer_kernel, static_cast<const uint4*>(src), static_cast<uint4*>(expert_out), n,
                           busy_cycles) != cudaSuccess) {
        cudaGetLastError();
        return MFR_ERR_LAUNCH;
    }
    return MFR_OK;
}
