// Host side of the C ABI declared in include/moe_finalize_rmsnorm.h:
// argument checks, variant choice, launch geometry, the plan's status word.
#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <new>

#include <cuda_runtime.h>

#include "moe_finalize_rmsnorm.h"
#include "mfr_internal.h"

struct mfr_plan_s {
    int64_t T;
    int64_t H;
    int64_t R;
    int k;
    int device;
    int sm_count;
    mfr_options opt;
    mfr::Launch launch;
    int* d_status;
    bool fused;        // residual + RMSNorm (false: moe_finalize_plan's plain finalize)
    bool fp4;          // made by moe_finalize_rmsnorm_nvfp4_plan: NVFP4 output
    bool expert_norm;  // made by moe_finalize_expert_rmsnorm_plan
    int sf_layout;     // NVFP4 plans: MFR_SF_ROW_MAJOR or MFR_SF_TILED_128x4
};

namespace {

thread_local char g_last_error[320] = "";

int fail(int code, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return code;
}

int fail_cuda(int code, const char* what, cudaError_t e) {
    return fail(code, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

// Half-open byte ranges [a, a+na) and [b, b+nb) share a byte.
bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}


}  // namespace

void mfr::set_last_error(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
}

extern "C" {

int moe_finalize_rmsnorm_supports(int64_t H, int k) {
    return (H >= 8 && H <= mfr::kMaxH && H % 8 == 0 && k >= 1 && k <= mfr::kMaxK) ? 1 : 0;
}

void moe_finalize_rmsnorm_default_options(mfr_options* opt) {
    if (!opt) return;
    opt->enable_pdl = 1;
    opt->force_variant = MFR_VARIANT_AUTO;
    opt->cluster_size = 0;
    opt->debug_checks = 0;
    opt->sentinel_skip = 0;
}

}  // extern "C"


namespace {

// Shared by the fused plan (residual + RMSNorm) and the plain-finalize plan.
int make_plan(mfr_plan_t* plan, int64_t T, int64_t H, int k, int64_t R, const mfr_options* opt,
              bool fused, bool fp4, bool expert_norm = false, int sf_layout = MFR_SF_ROW_MAJOR) {
    g_last_error[0] = '\0';
    if (!plan) return fail(MFR_ERR_INVALID_ARG, "plan must not be NULL");
    *plan = nullptr;
    if (T < 0 || R < 0) return fail(MFR_ERR_INVALID_ARG, "T and R must be >= 0 (T=%lld R=%lld)",
                                    (long long)T, (long long)R);
    if (!moe_finalize_rmsnorm_supports(H, k))
        return fail(MFR_ERR_UNSUPPORTED_SHAPE,
                    "unsupported shape H=%lld k=%d (need H %% 8 == 0, 8 <= H <= %d, 1 <= k <= %d)",
                    (long long)H, k, mfr::kMaxH, mfr::kMaxK);
    if (R > INT32_MAX) return fail(MFR_ERR_UNSUPPORTED_SHAPE, "R must fit an int32 index");
    if (T > (int64_t(1) << 26))
        return fail(MFR_ERR_UNSUPPORTED_SHAPE, "T=%lld exceeds 2^26 tokens per call", (long long)T);

    mfr_options o;
    moe_finalize_rmsnorm_default_options(&o);
    if (opt) o = *opt;
    if (o.force_variant < MFR_VARIANT_AUTO || o.force_variant > MFR_VARIANT_STREAM)
        return fail(MFR_ERR_INVALID_ARG, "force_variant %d is not available", o.force_variant);
    if (!(o.cluster_size == 0 || o.cluster_size == 1 || o.cluster_size == 2 ||
          o.cluster_size == 4 || o.cluster_size == 8 || o.cluster_size == 16))
        return fail(MFR_ERR_INVALID_ARG, "cluster_size must be 0, 1, 2, 4, 8 or 16");

    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { cudaGetLastError(); return fail_cuda(MFR_ERR_BAD_DEVICE, "cudaGetDevice", e); }
    int major = 0, minor = 0, sms = 0, smem_optin = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) {
        cudaGetLastError();
        return fail_cuda(MFR_ERR_BAD_DEVICE, "cudaDeviceGetAttribute", e);
    }
    if (major != 10 || minor != 3)
        return fail(MFR_ERR_BAD_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a only",
                    dev, major, minor);

    // ring depth the bulk-copy kernel would get on this device: room is left
    // for the ring kernel's static shared memory (at most 1152 bytes, in its
    // NVFP4 form: the encode-scale table) and slack
    const int ring_budget = smem_optin - 2048;
    int stages = 0;
    while (stages < mfr::kMaxStages && mfr::stream_smem_bytes(k, stages + 1, fused) <= ring_budget) ++stages;

    mfr::PolicyIn in{T, H, k, fused, fp4, expert_norm, o.force_variant, o.cluster_size, stages, sms};
    mfr::PolicyOut pol{};
    char why[200] = "";
    const int prc = mfr::choose_launch(in, &pol, why, sizeof why, mfr::stream_threads());
    if (prc != MFR_OK) return fail(prc, "%s", why);

    mfr::Launch l{};
    l.pdl = o.enable_pdl ? 1 : 0;
    l.grid_y = 1;
    l.fused = fused ? 1 : 0;
    l.fp4 = fp4 ? 1 : 0;
    l.expert_norm = expert_norm ? 1 : 0;
    l.sf_tiled = (fp4 && sf_layout == MFR_SF_TILED_128x4) ? 1 : 0;
    l.all_slots = mfr::ring_all_slots(T, H, k, fused, fp4, expert_norm) ? 1 : 0;
    l.variant = pol.variant;
    l.early_trigger = pol.early_trigger;
    l.cluster = pol.cluster;
    l.cpt = pol.cpt;
    l.block = pol.block;
    l.grid_x = pol.grid_x;

    if (l.variant == MFR_VARIANT_STREAM) {
        l.stages = stages;
        l.smem_bytes = mfr::stream_smem_bytes(k, stages, fused);
        // the attribute is per kernel, shared by every plan: always the device
        // maximum, so a plan with a deeper ring never loses its setting
        if ((e = mfr::stream_prepare(static_cast<int>(H), fused, fp4, ring_budget, expert_norm, l.sf_tiled != 0,
                                     l.all_slots != 0)) !=
            cudaSuccess) {
            cudaGetLastError();
            return fail_cuda(MFR_ERR_CUDA, "kernel attribute setup", e);
        }
    } else {
        l.smem_bytes = 0;
        // Slot rows and weights in registers shorten the path from the
        // dependency wait to the data, unless the extra registers make the
        // grid take more waves of resident CTAs (512-thread CTAs fit twice
        // per SM without them, once with them).
        l.regslots = 1;
        auto waves = [&](int per_sm) -> int64_t {
            const int64_t slots = static_cast<int64_t>(per_sm) * sms;
            return slots > 0 ? (l.grid_x + slots - 1) / slots : INT64_MAX;
        };
        if (expert_norm) {
            // The one-pass form holds up to 8 rows of at most 2 chunks per
            // thread; one CTA per token takes the two-pass form instead where
            // the one-pass form's registers would add a wave of CTAs.
            l.regslots = mfr::expert_norm_one_pass(k, l.cpt) ? 1 : 0;
            if (l.regslots && l.cluster == 1) {
                int one = 0, two = 0;
                if ((e = mfr::expert_norm_blocks_per_sm(l, true, &one)) != cudaSuccess ||
                    (e = mfr::expert_norm_blocks_per_sm(l, false, &two)) != cudaSuccess) {
                    cudaGetLastError();
                    return fail_cuda(MFR_ERR_CUDA, "occupancy query", e);
                }
                if (two > 0 && waves(two) < waves(one)) l.regslots = 0;
            }
            if (l.cluster > 1 && !l.regslots)
                return fail(MFR_ERR_UNSUPPORTED_SHAPE, "no per-expert RMSNorm cluster form for k=%d, H=%lld",
                            k, (long long)H);
            if ((e = mfr::expert_norm_prepare(l)) != cudaSuccess) {
                cudaGetLastError();
                return fail_cuda(MFR_ERR_CUDA, "kernel attribute setup", e);
            }
        } else {
            int with_regs = 0, without = 0;
            if ((e = mfr::rows_blocks_per_sm(l, true, &with_regs)) != cudaSuccess ||
                (e = mfr::rows_blocks_per_sm(l, false, &without)) != cudaSuccess) {
                cudaGetLastError();
                return fail_cuda(MFR_ERR_CUDA, "occupancy query", e);
            }
            if (without > 0 && waves(without) < waves(with_regs)) l.regslots = 0;
        }
        l.prefetch_out = (fused && l.cpt == 1 && l.regslots && T * H <= mfr::kPrefetchOutMaxElems) ? 1 : 0;
        if (!expert_norm && (e = mfr::rows_prepare(l)) != cudaSuccess) {
            cudaGetLastError();
            return fail_cuda(MFR_ERR_CUDA, "kernel attribute setup", e);
        }
        if (l.cluster > 1 && (fused || expert_norm)) {
            int nclusters = 0;
            e = expert_norm ? mfr::expert_norm_max_active_clusters(l, &nclusters)
                            : mfr::rows_max_active_clusters(l, &nclusters);
            if (e != cudaSuccess || nclusters < 1) {
                cudaGetLastError();
                return fail(MFR_ERR_UNSUPPORTED_SHAPE, "a cluster of %d CTAs x %d threads cannot be resident",
                            l.cluster, l.block);
            }
        }
    }

    int* status = nullptr;
    if ((e = cudaMalloc(&status, sizeof(int))) != cudaSuccess) {
        cudaGetLastError();
        return fail_cuda(MFR_ERR_CUDA, "cudaMalloc(status)", e);
    }
    if ((e = cudaMemset(status, 0, sizeof(int))) != cudaSuccess) {
        cudaFree(status);
        cudaGetLastError();
        return fail_cuda(MFR_ERR_CUDA, "cudaMemset(status)", e);
    }
    mfr_plan_s* p = new (std::nothrow) mfr_plan_s{};
    if (!p) {
        cudaFree(status);
        return fail(MFR_ERR_CUDA, "out of host memory");
    }
    p->T = T;
    p->H = H;
    p->R = R;
    p->k = k;
    p->device = dev;
    p->sm_count = sms;
    p->opt = o;
    p->launch = l;
    p->d_status = status;
    p->fused = fused;
    p->fp4 = fp4;
    p->expert_norm = expert_norm;
    p->sf_layout = sf_layout;
    *plan = p;
    return MFR_OK;
}

}  // namespace

extern "C" {

int moe_finalize_rmsnorm_plan(mfr_plan_t* plan, int64_t T, int64_t H, int k, int64_t R,
                              const mfr_options* opt) {
    return make_plan(plan, T, H, k, R, opt, true, false);
}

int moe_finalize_rmsnorm_nvfp4_plan(mfr_plan_t* plan, int64_t T, int64_t H, int k, int64_t R,
                                    const mfr_options* opt) {
    return make_plan(plan, T, H, k, R, opt, true, true);
}

int moe_finalize_rmsnorm_nvfp4_plan_ex(mfr_plan_t* plan, int64_t T, int64_t H, int k, int64_t R,
                                       const mfr_options* opt, int sf_layout) {
    if (sf_layout != MFR_SF_ROW_MAJOR && sf_layout != MFR_SF_TILED_128x4) {
        if (plan) *plan = nullptr;
        return fail(MFR_ERR_INVALID_ARG, "sf_layout %d is not MFR_SF_ROW_MAJOR or MFR_SF_TILED_128x4", sf_layout);
    }
    return make_plan(plan, T, H, k, R, opt, true, true, false, sf_layout);
}

int64_t moe_finalize_rmsnorm_nvfp4_sf_bytes(mfr_plan_t plan) {
    if (!plan || !plan->fp4) return -1;
    const int64_t S = plan->H / 16;
    if (plan->sf_layout == MFR_SF_TILED_128x4)
        return (plan->T + 127) / 128 * 128 * ((S + 3) / 4 * 4);
    return plan->T * S;
}

int moe_finalize_plan(mfr_plan_t* plan, int64_t T, int64_t H, int k, int64_t R, const mfr_options* opt) {
    return make_plan(plan, T, H, k, R, opt, false, false);
}

int moe_finalize_expert_rmsnorm_plan(mfr_plan_t* plan, int64_t T, int64_t H, int k, int64_t R,
                                     const mfr_options* opt) {
    return make_plan(plan, T, H, k, R, opt, false, false, true);
}

int moe_finalize_expert_rmsnorm_run(mfr_plan_t plan, const void* expert_out, const int32_t* permuted_row_of,
                                    const float* topk_weights, const void* gamma, float eps, void* out,
                                    void* stream) {
    g_last_error[0] = '\0';
    if (!plan) return fail(MFR_ERR_INVALID_ARG, "plan must not be NULL");
    if (!plan->expert_norm)
        return fail(MFR_ERR_INVALID_ARG, "this plan was not made by moe_finalize_expert_rmsnorm_plan");
    const int64_t T = plan->T, H = plan->H, R = plan->R;
    const int k = plan->k;
    if (T == 0) return MFR_OK;
    if (!permuted_row_of || !topk_weights || !gamma || !out || (R > 0 && !expert_out))
        return fail(MFR_ERR_INVALID_ARG, "a required pointer is NULL");
    if (!std::isfinite(eps) || eps < 0.f)
        return fail(MFR_ERR_INVALID_ARG, "eps must be finite and >= 0");
    if (!aligned(expert_out, 16) || !aligned(gamma, 16) || !aligned(out, 16))
        return fail(MFR_ERR_MISALIGNED, "expert_out, gamma and out must be 16-byte aligned");
    if (!aligned(permuted_row_of, 4) || !aligned(topk_weights, 4))
        return fail(MFR_ERR_MISALIGNED, "permuted_row_of and topk_weights must be 4-byte aligned");
    const size_t n_out = static_cast<size_t>(T * H) * 2;
    const size_t n_e = static_cast<size_t>(R * H) * 2;
    const size_t n_tk = static_cast<size_t>(T * k) * 4;
    if (overlaps(out, n_out, expert_out, n_e) || overlaps(out, n_out, permuted_row_of, n_tk) ||
        overlaps(out, n_out, topk_weights, n_tk) || overlaps(out, n_out, gamma, static_cast<size_t>(H) * 2))
        return fail(MFR_ERR_INVALID_ARG, "out overlaps an input");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { cudaGetLastError(); return fail_cuda(MFR_ERR_CUDA, "cudaGetDevice", e); }
    if (dev != plan->device)
        return fail(MFR_ERR_INVALID_ARG, "current device %d is not the plan's device %d", dev, plan->device);

    mfr::Params p{};
    p.expert_out = static_cast<const uint16_t*>(expert_out);
    p.permuted_row_of = permuted_row_of;
    p.topk_weights = topk_weights;
    p.gamma = static_cast<const uint16_t*>(gamma);
    p.out = static_cast<uint16_t*>(out);
    p.status = plan->d_status;
    p.T = T;
    p.R = R;
    p.H = static_cast<int>(H);
    p.k = k;
    p.eps = eps;
    p.sentinel = plan->opt.sentinel_skip ? 1 : 0;
    p.early_trigger = plan->launch.early_trigger;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    e = plan->launch.variant == MFR_VARIANT_STREAM ? mfr::stream_launch(p, plan->launch, s)
                                                   : mfr::expert_norm_launch(p, plan->launch, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail_cuda(MFR_ERR_LAUNCH, "kernel launch", e);
    }
    if (plan->opt.debug_checks) {
        int st = 0;
        const int rc = moe_finalize_rmsnorm_get_status(plan, stream, &st);
        if (rc != MFR_OK) return rc;
        if (st & MFR_STATUS_BAD_INDEX)
            return fail(MFR_ERR_BAD_INDEX, "a permuted_row_of entry was outside [0, %lld)", (long long)R);
    }
    return MFR_OK;
}

int moe_finalize_run(mfr_plan_t plan, const void* expert_out, const int32_t* permuted_row_of,
                     const float* topk_weights, void* out, void* stream) {
    g_last_error[0] = '\0';
    if (!plan) return fail(MFR_ERR_INVALID_ARG, "plan must not be NULL");
    if (plan->fused) return fail(MFR_ERR_INVALID_ARG, "this plan was made by moe_finalize_rmsnorm_plan");
    if (plan->expert_norm)
        return fail(MFR_ERR_INVALID_ARG, "this plan was made by moe_finalize_expert_rmsnorm_plan");
    const int64_t T = plan->T, H = plan->H, R = plan->R;
    const int k = plan->k;
    if (T == 0) return MFR_OK;
    if (!permuted_row_of || !topk_weights || !out || (R > 0 && !expert_out))
        return fail(MFR_ERR_INVALID_ARG, "a required pointer is NULL");
    if (!aligned(expert_out, 16) || !aligned(out, 16))
        return fail(MFR_ERR_MISALIGNED, "expert_out and out must be 16-byte aligned");
    if (!aligned(permuted_row_of, 4) || !aligned(topk_weights, 4))
        return fail(MFR_ERR_MISALIGNED, "permuted_row_of and topk_weights must be 4-byte aligned");
    const size_t n_out = static_cast<size_t>(T * H) * 2;
    const size_t n_e = static_cast<size_t>(R * H) * 2;
    const size_t n_tk = static_cast<size_t>(T * k) * 4;
    if (overlaps(out, n_out, expert_out, n_e) || overlaps(out, n_out, permuted_row_of, n_tk) ||
        overlaps(out, n_out, topk_weights, n_tk))
        return fail(MFR_ERR_INVALID_ARG, "out overlaps an input");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { cudaGetLastError(); return fail_cuda(MFR_ERR_CUDA, "cudaGetDevice", e); }
    if (dev != plan->device)
        return fail(MFR_ERR_INVALID_ARG, "current device %d is not the plan's device %d", dev, plan->device);

    mfr::Params p{};
    p.expert_out = static_cast<const uint16_t*>(expert_out);
    p.permuted_row_of = permuted_row_of;
    p.topk_weights = topk_weights;
    p.out = static_cast<uint16_t*>(out);
    p.status = plan->d_status;
    p.T = T;
    p.R = R;
    p.H = static_cast<int>(H);
    p.k = k;
    p.sentinel = plan->opt.sentinel_skip ? 1 : 0;
    p.early_trigger = plan->launch.early_trigger;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    e = plan->launch.variant == MFR_VARIANT_STREAM ? mfr::stream_launch(p, plan->launch, s)
                                                   : mfr::rows_launch(p, plan->launch, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail_cuda(MFR_ERR_LAUNCH, "kernel launch", e);
    }
    if (plan->opt.debug_checks) {
        int st = 0;
        const int rc = moe_finalize_rmsnorm_get_status(plan, stream, &st);
        if (rc != MFR_OK) return rc;
        if (st & MFR_STATUS_TIMEOUT)
            return fail(MFR_ERR_CUDA, "an on-chip wait timed out; the outputs are not valid");
        if (st & MFR_STATUS_BAD_INDEX)
            return fail(MFR_ERR_BAD_INDEX, "a permuted_row_of entry was outside [0, %lld)", (long long)R);
    }
    return MFR_OK;
}

}  // extern "C"

namespace {

// Checks and launches one fused call: bf16 output (out) or NVFP4 output
// (out_q, out_sf, s_enc) according to the plan.
int fused_run(mfr_plan_t plan, const void* expert_out, const int32_t* permuted_row_of,
              const float* topk_weights, const float* residual_in, float* residual_out, const void* gamma,
              float eps, void* out, void* out_q, void* out_sf, float s_enc, void* stream) {
    const int64_t T = plan->T, H = plan->H, R = plan->R;
    const int k = plan->k;
    if (T == 0) return MFR_OK;
    const bool fp4 = plan->fp4;
    if (!permuted_row_of || !topk_weights || !residual_in || !residual_out || !gamma ||
        (fp4 ? (!out_q || !out_sf) : !out) || (R > 0 && !expert_out))
        return fail(MFR_ERR_INVALID_ARG, "a required pointer is NULL");
    if (!std::isfinite(eps) || eps < 0.f)
        return fail(MFR_ERR_INVALID_ARG, "eps must be finite and >= 0");
    if (fp4 && (!std::isfinite(s_enc) || s_enc <= 0.f))
        return fail(MFR_ERR_INVALID_ARG, "the NVFP4 tensor scale must be finite and > 0");
    if (!aligned(expert_out, 16) || !aligned(residual_in, 16) || !aligned(residual_out, 16) ||
        !aligned(gamma, 16) || (!fp4 && !aligned(out, 16)))
        return fail(MFR_ERR_MISALIGNED, "expert_out, residual_in, residual_out, gamma and out must be "
                                        "16-byte aligned");
    if (!aligned(permuted_row_of, 4) || !aligned(topk_weights, 4) || (fp4 && !aligned(out_q, 4)))
        return fail(MFR_ERR_MISALIGNED, "permuted_row_of, topk_weights and out_q must be 4-byte aligned");

    const size_t n_res = static_cast<size_t>(T * H) * sizeof(float);
    const size_t n_out = static_cast<size_t>(T * H) * 2;
    const size_t n_e = static_cast<size_t>(R * H) * 2;
    const size_t n_tk = static_cast<size_t>(T * k) * 4;
    if (residual_out != residual_in && overlaps(residual_out, n_res, residual_in, n_res))
        return fail(MFR_ERR_INVALID_ARG, "residual_out partially overlaps residual_in");
    if (overlaps(residual_out, n_res, expert_out, n_e) || overlaps(residual_out, n_res, permuted_row_of, n_tk) ||
        overlaps(residual_out, n_res, topk_weights, n_tk) || overlaps(residual_out, n_res, gamma, H * 2))
        return fail(MFR_ERR_INVALID_ARG, "residual_out overlaps an input");
    // every output region against every other argument
    const void* outs[2] = {fp4 ? out_q : out, fp4 ? out_sf : nullptr};
    const size_t out_bytes[2] = {fp4 ? n_out / 4 : n_out,
                                 fp4 ? static_cast<size_t>(moe_finalize_rmsnorm_nvfp4_sf_bytes(plan)) : 0};
    for (int o = 0; o < 2; ++o) {
        if (!outs[o]) continue;
        if (overlaps(outs[o], out_bytes[o], expert_out, n_e) || overlaps(outs[o], out_bytes[o], permuted_row_of, n_tk) ||
            overlaps(outs[o], out_bytes[o], topk_weights, n_tk) || overlaps(outs[o], out_bytes[o], residual_in, n_res) ||
            overlaps(outs[o], out_bytes[o], residual_out, n_res) || overlaps(outs[o], out_bytes[o], gamma, H * 2))
            return fail(MFR_ERR_INVALID_ARG, "an output overlaps another argument");
    }
    if (fp4 && overlaps(out_q, out_bytes[0], out_sf, out_bytes[1]))
        return fail(MFR_ERR_INVALID_ARG, "out_q and out_sf overlap");

    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { cudaGetLastError(); return fail_cuda(MFR_ERR_CUDA, "cudaGetDevice", e); }
    if (dev != plan->device)
        return fail(MFR_ERR_INVALID_ARG, "current device %d is not the plan's device %d", dev, plan->device);

    mfr::Params p{};
    p.expert_out = static_cast<const uint16_t*>(expert_out);
    p.permuted_row_of = permuted_row_of;
    p.topk_weights = topk_weights;
    p.residual_in = residual_in;
    p.residual_out = residual_out;
    p.gamma = static_cast<const uint16_t*>(gamma);
    p.out = static_cast<uint16_t*>(out);
    p.out_q = static_cast<uint8_t*>(out_q);
    p.out_sf = static_cast<uint8_t*>(out_sf);
    p.s_enc = s_enc;
    p.status = plan->d_status;
    p.T = T;
    p.R = R;
    p.H = static_cast<int>(H);
    p.k = k;
    p.eps = eps;
    p.sentinel = plan->opt.sentinel_skip ? 1 : 0;
    p.early_trigger = plan->launch.early_trigger;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    e = plan->launch.variant == MFR_VARIANT_STREAM ? mfr::stream_launch(p, plan->launch, s)
                                                   : mfr::rows_launch(p, plan->launch, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail_cuda(MFR_ERR_LAUNCH, "kernel launch", e);
    }
    if (plan->opt.debug_checks) {
        int st = 0;
        const int rc = moe_finalize_rmsnorm_get_status(plan, stream, &st);
        if (rc != MFR_OK) return rc;
        if (st & MFR_STATUS_TIMEOUT)
            return fail(MFR_ERR_CUDA, "an on-chip wait timed out; the outputs are not valid");
        if (st & MFR_STATUS_BAD_INDEX)
            return fail(MFR_ERR_BAD_INDEX, "a permuted_row_of entry was outside [0, %lld)", (long long)R);
    }
    return MFR_OK;
}

}  // namespace

extern "C" {

int moe_finalize_rmsnorm_run(mfr_plan_t plan, const void* expert_out, const int32_t* permuted_row_of,
                             const float* topk_weights, const float* residual_in, float* residual_out,
                             const void* gamma, float eps, void* out, void* stream) {
    g_last_error[0] = '\0';
    if (!plan) return fail(MFR_ERR_INVALID_ARG, "plan must not be NULL");
    if (!plan->fused || plan->fp4)
        return fail(MFR_ERR_INVALID_ARG, "this plan was not made by moe_finalize_rmsnorm_plan");
    return fused_run(plan, expert_out, permuted_row_of, topk_weights, residual_in, residual_out, gamma, eps, out,
                     nullptr, nullptr, 0.f, stream);
}

int moe_finalize_rmsnorm_nvfp4_run(mfr_plan_t plan, const void* expert_out, const int32_t* permuted_row_of,
                                   const float* topk_weights, const float* residual_in, float* residual_out,
                                   const void* gamma, float eps, float s_enc, void* out_q, void* out_sf,
                                   void* stream) {
    g_last_error[0] = '\0';
    if (!plan) return fail(MFR_ERR_INVALID_ARG, "plan must not be NULL");
    if (!plan->fp4) return fail(MFR_ERR_INVALID_ARG, "this plan was not made by moe_finalize_rmsnorm_nvfp4_plan");
    return fused_run(plan, expert_out, permuted_row_of, topk_weights, residual_in, residual_out, gamma, eps,
                     nullptr, out_q, out_sf, s_enc, stream);
}

}  // extern "C"

namespace {

// Device workspace of run_host: every tensor of one call, each 256-byte aligned.
struct HostLayout {
    size_t e, idx, w, res_in, res_out, gamma, out, total;
};

size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

HostLayout host_layout(const mfr_plan_s* p) {
    HostLayout l{};
    size_t off = 0;
    auto take = [&](size_t bytes) { const size_t at = off; off += align256(bytes); return at; };
    l.e = take(static_cast<size_t>(p->R * p->H) * 2);
    l.idx = take(static_cast<size_t>(p->T * p->k) * 4);
    l.w = take(static_cast<size_t>(p->T * p->k) * 4);
    l.res_in = take(static_cast<size_t>(p->T * p->H) * 4);
    l.res_out = take(static_cast<size_t>(p->T * p->H) * 4);
    l.gamma = take(static_cast<size_t>(p->H) * 2);
    l.out = take(static_cast<size_t>(p->T * p->H) * 2);
    l.total = off;
    return l;
}

}  // namespace

extern "C" {

int64_t moe_finalize_rmsnorm_host_workspace_bytes(mfr_plan_t plan) {
    if (!plan || !plan->fused || plan->fp4) return -1;
    return static_cast<int64_t>(host_layout(plan).total);
}

int moe_finalize_rmsnorm_run_host(mfr_plan_t plan, const void* h_expert_out, const int32_t* h_permuted_row_of,
                                  const float* h_topk_weights, const float* h_residual_in, float* h_residual_out,
                                  const void* h_gamma, float eps, void* h_out, void* d_workspace,
                                  int64_t workspace_bytes, void* stream) {
    g_last_error[0] = '\0';
    if (!plan) return fail(MFR_ERR_INVALID_ARG, "plan must not be NULL");
    if (!plan->fused || plan->fp4)
        return fail(MFR_ERR_INVALID_ARG, "this plan was not made by moe_finalize_rmsnorm_plan");
    if (plan->T == 0) return MFR_OK;
    const HostLayout L = host_layout(plan);
    if (!d_workspace || workspace_bytes < static_cast<int64_t>(L.total))
        return fail(MFR_ERR_INVALID_ARG, "workspace of %lld bytes is smaller than the %llu the plan needs",
                    (long long)workspace_bytes, (unsigned long long)L.total);
    if (!aligned(d_workspace, 256)) return fail(MFR_ERR_MISALIGNED, "the workspace must be 256-byte aligned");
    if (!h_permuted_row_of || !h_topk_weights || !h_residual_in || !h_residual_out || !h_gamma || !h_out ||
        (plan->R > 0 && !h_expert_out))
        return fail(MFR_ERR_INVALID_ARG, "a required host pointer is NULL");
    const int64_t T = plan->T, H = plan->H, R = plan->R;
    const int k = plan->k;
    unsigned char* ws = static_cast<unsigned char*>(d_workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    struct Copy { void* dst; const void* src; size_t bytes; cudaMemcpyKind kind; };
    const Copy in[] = {
        {ws + L.e, h_expert_out, static_cast<size_t>(R * H) * 2, cudaMemcpyHostToDevice},
        {ws + L.idx, h_permuted_row_of, static_cast<size_t>(T * k) * 4, cudaMemcpyHostToDevice},
        {ws + L.w, h_topk_weights, static_cast<size_t>(T * k) * 4, cudaMemcpyHostToDevice},
        {ws + L.res_in, h_residual_in, static_cast<size_t>(T * H) * 4, cudaMemcpyHostToDevice},
        {ws + L.gamma, h_gamma, static_cast<size_t>(H) * 2, cudaMemcpyHostToDevice},
    };
    for (const Copy& c : in) {
        if (c.bytes == 0) continue;
        const cudaError_t e = cudaMemcpyAsync(c.dst, c.src, c.bytes, c.kind, s);
        if (e != cudaSuccess) { cudaGetLastError(); return fail_cuda(MFR_ERR_CUDA, "host-to-device copy", e); }
    }
    const int rc = moe_finalize_rmsnorm_run(plan, R > 0 ? ws + L.e : nullptr,
                                            reinterpret_cast<const int32_t*>(ws + L.idx),
                                            reinterpret_cast<const float*>(ws + L.w),
                                            reinterpret_cast<const float*>(ws + L.res_in),
                                            reinterpret_cast<float*>(ws + L.res_out), ws + L.gamma, eps,
                                            ws + L.out, stream);
    if (rc != MFR_OK) return rc;
    const Copy outc[] = {
        {h_residual_out, ws + L.res_out, static_cast<size_t>(T * H) * 4, cudaMemcpyDeviceToHost},
        {h_out, ws + L.out, static_cast<size_t>(T * H) * 2, cudaMemcpyDeviceToHost},
    };
    for (const Copy& c : outc) {
        const cudaError_t e = cudaMemcpyAsync(c.dst, c.src, c.bytes, c.kind, s);
        if (e != cudaSuccess) { cudaGetLastError(); return fail_cuda(MFR_ERR_CUDA, "device-to-host copy", e); }
    }
    return MFR_OK;
}

int moe_finalize_rmsnorm_get_status(mfr_plan_t plan, void* stream, int* device_status) {
    g_last_error[0] = '\0';
    if (!plan || !device_status) return fail(MFR_ERR_INVALID_ARG, "plan and device_status must not be NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int h = 0;
    cudaError_t e = cudaMemcpyAsync(&h, plan->d_status, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemsetAsync(plan->d_status, 0, sizeof(int), s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail_cuda(MFR_ERR_CUDA, "reading the status word", e);
    }
    *device_status = h;
    return MFR_OK;
}

int moe_finalize_rmsnorm_wait_selftest(mfr_plan_t plan, int64_t limit_cycles, int arrive, void* stream) {
    g_last_error[0] = '\0';
    if (!plan) return fail(MFR_ERR_INVALID_ARG, "plan must not be NULL");
    if (limit_cycles < 1 || limit_cycles > (int64_t(1) << 32))
        return fail(MFR_ERR_INVALID_ARG, "limit_cycles must be in [1, 2^32] (got %lld)", (long long)limit_cycles);
    const cudaError_t e = mfr::wait_selftest_launch(plan->d_status, static_cast<long long>(limit_cycles),
                                                    arrive ? 1 : 0, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail_cuda(MFR_ERR_LAUNCH, "self-test kernel launch", e);
    }
    return MFR_OK;
}

int moe_finalize_rmsnorm_launch_floor(mfr_plan_t plan, void* stream) {
    g_last_error[0] = '\0';
    if (!plan) return fail(MFR_ERR_INVALID_ARG, "plan must not be NULL");
    if (plan->T == 0) return MFR_OK;
    const cudaError_t e = mfr::floor_launch(plan->d_status, plan->launch, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail_cuda(MFR_ERR_LAUNCH, "floor kernel launch", e);
    }
    return MFR_OK;
}

int moe_finalize_rmsnorm_launch_floor_work(mfr_plan_t plan, int work, const void* expert_out,
                                           const int32_t* permuted_row_of, const float* residual_in,
                                           float* residual_out, void* out, void* stream) {
    g_last_error[0] = '\0';
    if (!plan) return fail(MFR_ERR_INVALID_ARG, "plan must not be NULL");
    if (work < 0 || work > (MFR_FLOOR_LOAD | MFR_FLOOR_EXCHANGE | MFR_FLOOR_STORE))
        return fail(MFR_ERR_INVALID_ARG, "work must be a combination of the MFR_FLOOR_* bits (got %d)", work);
    if (!plan->fused || plan->fp4 || plan->expert_norm)
        return fail(MFR_ERR_INVALID_ARG, "the work floor takes plans made by moe_finalize_rmsnorm_plan");
    if (plan->launch.variant == MFR_VARIANT_STREAM)
        return fail(MFR_ERR_UNSUPPORTED_SHAPE, "the work floor covers the cluster and one-CTA-per-token variants");
    const int64_t T = plan->T, H = plan->H, R = plan->R;
    const int k = plan->k;
    if (T == 0) return MFR_OK;
    const bool load = work & MFR_FLOOR_LOAD, store = work & MFR_FLOOR_STORE;
    if (!permuted_row_of || (load && (!residual_in || (R > 0 && !expert_out))) ||
        (store && (!residual_out || !out)))
        return fail(MFR_ERR_INVALID_ARG, "a pointer the requested work needs is NULL");
    if (!aligned(permuted_row_of, 4) || (load && (!aligned(expert_out, 16) || !aligned(residual_in, 16))) ||
        (store && (!aligned(residual_out, 16) || !aligned(out, 16))))
        return fail(MFR_ERR_MISALIGNED, "misaligned pointer");
    const size_t n_res = static_cast<size_t>(T * H) * 4, n_out = static_cast<size_t>(T * H) * 2;
    const size_t n_e = static_cast<size_t>(R * H) * 2, n_tk = static_cast<size_t>(T * k) * 4;
    if (store && (overlaps(residual_out, n_res, out, n_out) || overlaps(out, n_out, permuted_row_of, n_tk) ||
                  overlaps(residual_out, n_res, permuted_row_of, n_tk) ||
                  (load && (overlaps(out, n_out, expert_out, n_e) || overlaps(out, n_out, residual_in, n_res) ||
                            overlaps(residual_out, n_res, expert_out, n_e) ||
                            (residual_out != residual_in && overlaps(residual_out, n_res, residual_in, n_res))))))
        return fail(MFR_ERR_INVALID_ARG, "an output overlaps another argument");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { cudaGetLastError(); return fail_cuda(MFR_ERR_CUDA, "cudaGetDevice", e); }
    if (dev != plan->device)
        return fail(MFR_ERR_INVALID_ARG, "current device %d is not the plan's device %d", dev, plan->device);
    mfr::Params p{};
    p.expert_out = static_cast<const uint16_t*>(expert_out);
    p.permuted_row_of = permuted_row_of;
    p.residual_in = residual_in;
    p.residual_out = residual_out;
    p.out = static_cast<uint16_t*>(out);
    p.status = plan->d_status;
    p.T = T;
    p.R = R;
    p.H = static_cast<int>(H);
    p.k = k;
    p.early_trigger = plan->launch.early_trigger;
    e = mfr::floor_work_launch(p, plan->launch, work, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail_cuda(MFR_ERR_LAUNCH, "floor kernel launch", e);
    }
    return MFR_OK;
}

int moe_finalize_rmsnorm_plan_info(mfr_plan_t plan, mfr_plan_info* info) {
    if (!plan || !info) return fail(MFR_ERR_INVALID_ARG, "plan and info must not be NULL");
    const mfr::Launch& l = plan->launch;
    info->variant = l.variant;
    info->grid_x = l.grid_x;
    info->grid_y = l.grid_y;
    info->block = l.block;
    info->cluster = l.cluster;
    info->smem_bytes = l.smem_bytes;
    info->chunks_per_thread = l.cpt;
    info->sm_count = plan->sm_count;
    info->slot_registers = l.regslots;
    return MFR_OK;
}

void moe_finalize_rmsnorm_destroy(mfr_plan_t plan) {
    if (!plan) return;
    if (plan->d_status) {
        cudaFree(plan->d_status);
        cudaGetLastError();
    }
    delete plan;
}

const char* moe_finalize_rmsnorm_strerror(int code) {
    switch (code) {
        case MFR_OK: return "ok";
        case MFR_ERR_INVALID_ARG: return "invalid argument";
        case MFR_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case MFR_ERR_MISALIGNED: return "misaligned pointer";
        case MFR_ERR_BAD_DEVICE: return "unsupported or unavailable device (needs sm_103)";
        case MFR_ERR_LAUNCH: return "kernel launch failed";
        case MFR_ERR_CUDA: return "CUDA runtime error";
        case MFR_ERR_BAD_INDEX: return "permuted_row_of entry out of range";
        default: return "unknown error code";
    }
}

const char* moe_finalize_rmsnorm_last_error(void) { return g_last_error; }

}  // extern "C"
