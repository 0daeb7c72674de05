// moe_finalize_rmsnorm_run_noalloc: the fused path for callers that cannot
// allocate device memory.
//
// The planned path (moe_finalize_rmsnorm_plan) allocates one device word per
// plan with cudaMalloc for the kernel's status flags.  Some callers cannot do
// that: engines that own every byte of device memory through their own pool
// and forbid allocations outside it (so memory accounting stays exact and a
// late out-of-memory cannot happen mid-request), and hosts that embed the
// kernel where cudaMalloc's implicit synchronisation and latency are not
// allowed on the request path.  This entry point needs no plan and allocates
// nothing: the status words live in a file-scope __device__ array that every
// GPU loading the library holds until the process exits.
//
// It always launches the persistent bulk-copy kernel (stream_kernel), with the
// same geometry rules as a planned MFR_VARIANT_STREAM call.
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "moe_finalize_rmsnorm.h"
#include "mfr_internal.h"

namespace {

// Scratch of the allocation-free path: one status word per slot.
static __device__ __align__(256) int g_noalloc_status[MFR_NOALLOC_SLOTS];

constexpr int kMaxDevices = 64;
constexpr int kMaxStagesNoAlloc = 8;

struct DeviceSetup {
    bool ready;
    int* status;       // device address of g_noalloc_status on this device
    int sms;
    int ring_budget;   // dynamic shared memory the ring may use
};

std::mutex g_setup_lock;
DeviceSetup g_setup[kMaxDevices];

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// Once per device, with that device current: the scratch array's device
// address (host code cannot use the symbol itself), the SM count and the
// kernel's shared-memory attribute.
int setup_device(int dev, DeviceSetup* out) {
    std::lock_guard<std::mutex> g(g_setup_lock);
    DeviceSetup& s = g_setup[dev];
    if (!s.ready) {
        int major = 0, minor = 0, sms = 0, optin = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
            cudaGetLastError();
            return MFR_ERR_BAD_DEVICE;
        }
        if (major != 10 || minor != 3) return MFR_ERR_BAD_DEVICE;
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_noalloc_status) != cudaSuccess || addr == nullptr) {
            cudaGetLastError();
            return MFR_ERR_CUDA;
        }
        // the same budget as the planned path (mfr_api.cu), so whichever sets
        // the per-kernel attribute last, every ring either path picks fits it
        const int budget = optin - 2048;
        // one attribute per kernel instantiation (by column tiles per token),
        // set to the device maximum exactly as the planned path sets it
        for (int h : {4096, 8192, 16384}) {
            if (mfr::stream_prepare(h, true, false, budget) != cudaSuccess ||
                (h <= 8192 && mfr::stream_prepare(h, true, false, budget, false, false, true) != cudaSuccess)) {
                cudaGetLastError();
                return MFR_ERR_CUDA;
            }
        }
        // start every slot at zero once, here, so no memset sits between the
        // producing kernel and a later call (it would cost the dependent
        // launch its overlap); after that a word is cleared only when a call
        // reads it back
        if (cudaMemset(addr, 0, sizeof(int) * MFR_NOALLOC_SLOTS) != cudaSuccess ||
            cudaDeviceSynchronize() != cudaSuccess) {
            cudaGetLastError();
            return MFR_ERR_CUDA;
        }
        s.status = static_cast<int*>(addr);
        s.sms = sms;
        s.ring_budget = budget;
        s.ready = true;
    }
    *out = s;
    return MFR_OK;
}

}  // namespace

extern "C" int moe_finalize_rmsnorm_run_noalloc(
    int64_t T, int64_t H, int k, int64_t R, const void* expert_out, const int32_t* permuted_row_of,
    const float* topk_weights, const float* residual_in, float* residual_out, const void* gamma, float eps,
    void* out, int slot, int* host_status, void* stream)
{
    mfr::set_last_error("");
    if (T < 0 || R < 0 || R > INT32_MAX || T > (int64_t(1) << 26))
        return mfr::set_last_error("T must be in [0, 2^26] and R in [0, 2^31)"), MFR_ERR_INVALID_ARG;
    if (!moe_finalize_rmsnorm_supports(H, k))
        return mfr::set_last_error("unsupported shape H=%lld k=%d", (long long)H, k), MFR_ERR_UNSUPPORTED_SHAPE;
    if (slot < 0 || slot >= MFR_NOALLOC_SLOTS)
        return mfr::set_last_error("slot %d is beyond the %d status words of the allocation-free scratch",
                                   slot, MFR_NOALLOC_SLOTS), MFR_ERR_INVALID_ARG;
    if (T == 0) {
        if (host_status) *host_status = 0;
        return MFR_OK;
    }
    if (!permuted_row_of || !topk_weights || !residual_in || !residual_out || !gamma || !out ||
        (R > 0 && !expert_out))
        return mfr::set_last_error("a required pointer is NULL"), MFR_ERR_INVALID_ARG;
    if (!std::isfinite(eps) || eps < 0.f)
        return mfr::set_last_error("eps must be finite and >= 0"), MFR_ERR_INVALID_ARG;
    if (!aligned(expert_out, 16) || !aligned(residual_in, 16) || !aligned(residual_out, 16) ||
        !aligned(gamma, 16) || !aligned(out, 16) || !aligned(permuted_row_of, 4) || !aligned(topk_weights, 4))
        return mfr::set_last_error("misaligned pointer"), MFR_ERR_MISALIGNED;
    const size_t n_res = static_cast<size_t>(T * H) * 4, n_out = static_cast<size_t>(T * H) * 2;
    const size_t n_e = static_cast<size_t>(R * H) * 2, n_tk = static_cast<size_t>(T * k) * 4;
    if (residual_out != residual_in && overlaps(residual_out, n_res, residual_in, n_res)) return MFR_ERR_INVALID_ARG;
    if (overlaps(residual_out, n_res, expert_out, n_e) || overlaps(residual_out, n_res, permuted_row_of, n_tk) ||
        overlaps(residual_out, n_res, topk_weights, n_tk) || overlaps(residual_out, n_res, gamma, H * 2) ||
        overlaps(out, n_out, expert_out, n_e) || overlaps(out, n_out, permuted_row_of, n_tk) ||
        overlaps(out, n_out, topk_weights, n_tk) || overlaps(out, n_out, residual_in, n_res) ||
        overlaps(out, n_out, residual_out, n_res) || overlaps(out, n_out, gamma, H * 2))
        return mfr::set_last_error("an output overlaps another argument"), MFR_ERR_INVALID_ARG;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return MFR_ERR_BAD_DEVICE; }
    if (dev < 0 || dev >= kMaxDevices) return MFR_ERR_BAD_DEVICE;
    DeviceSetup ds;
    const int rc = setup_device(dev, &ds);
    if (rc != MFR_OK)
        return mfr::set_last_error("set-up of device %d failed (needs sm_103)", dev), rc;

    int stages = 0;
    while (stages < kMaxStagesNoAlloc && mfr::stream_smem_bytes(k, stages + 1, true) <= ds.ring_budget) ++stages;
    if (stages < 2) return mfr::set_last_error("k=%d leaves no room for 2 ring stages", k), MFR_ERR_UNSUPPORTED_SHAPE;

    mfr::Launch l{};
    l.variant = MFR_VARIANT_STREAM;
    l.grid_x = mfr::stream_grid(T, ds.sms);
    l.grid_y = 1;
    l.block = mfr::stream_threads();
    l.cluster = 1;
    l.cpt = 1;
    l.stages = stages;
    l.smem_bytes = mfr::stream_smem_bytes(k, stages, true);
    l.pdl = 1;
    l.fused = 1;
    l.all_slots = mfr::ring_all_slots(T, H, k, true, false, false) ? 1 : 0;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int* status = ds.status + slot;

    mfr::Params p{};
    p.expert_out = static_cast<const uint16_t*>(expert_out);
    p.permuted_row_of = permuted_row_of;
    p.topk_weights = topk_weights;
    p.residual_in = residual_in;
    p.residual_out = residual_out;
    p.gamma = static_cast<const uint16_t*>(gamma);
    p.out = static_cast<uint16_t*>(out);
    p.status = status;
    p.T = T;
    p.R = R;
    p.H = static_cast<int>(H);
    p.k = k;
    p.eps = eps;
    if (mfr::stream_launch(p, l, s) != cudaSuccess) { cudaGetLastError(); return MFR_ERR_LAUNCH; }

    if (host_status) {
        // read the word, then clear it behind the read, in stream order: the
        // next call on this slot starts from zero without a memset of its own
        int h = 0;
        if (cudaMemcpyAsync(&h, status, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
            cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess) {
            cudaGetLastError();
            return MFR_ERR_CUDA;
        }
        *host_status = h;
    }
    return MFR_OK;
}
