// Declarations shared by the host ABI (mfr_api.cu) and the kernel files.
// Not part of the public ABI; see include/moe_finalize_rmsnorm.h.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "mfr_policy.h"

namespace mfr {

// Everything a kernel needs for one call; passed by value.
struct Params {
    const uint16_t* expert_out;     // bf16 bits [R, H]
    const int32_t* permuted_row_of; // [T, k]
    const float* topk_weights;      // [T, k]
    const float* residual_in;       // [T, H]
    float* residual_out;            // [T, H]
    const uint16_t* gamma;          // bf16 bits [H]
    uint16_t* out;                  // bf16 bits [T, H]
    uint8_t* out_q;                 // NVFP4 codes [T, H/2] (NVFP4 plans)
    uint8_t* out_sf;                // NVFP4 block scales, E4M3: [T, H/16] row-major, or tiled (Launch::sf_tiled)
    float s_enc;                    // NVFP4 tensor scale
    int* status;                    // device status word (MFR_STATUS_* bits)
    int64_t T;
    int64_t R;
    int H;
    int k;
    float eps;
    int sentinel;                   // 1: a negative index is a skipped non-local slot, not an error
    int early_trigger;              // 1: signal dependents at kernel entry; 0: after the loads
};

// Launch geometry fixed by the plan.
struct Launch {
    int variant;      // MFR_VARIANT_*
    int grid_x;
    int grid_y;
    int block;
    int cluster;      // CTAs per cluster along x (1 = no cluster)
    int smem_bytes;   // dynamic shared memory
    int cpt;          // 16-byte chunks per thread per row
    int pdl;          // programmatic stream serialization
    int stages;       // MFR_VARIANT_STREAM: shared-memory ring depth
    int fused;        // 1: residual + RMSNorm; 0: plain finalize (out = bf16(sum))
    int fp4;          // 1: the normalised output is written as NVFP4 instead of bf16
    int early_trigger;  // 1: signal dependents at kernel entry (small grids only)
    int regslots;     // one-CTA-per-token kernels: slot rows/weights held in registers
    int expert_norm;  // 1: RMSNorm per expert row before the weighted sum (mfr_expert_norm.cu)
    int prefetch_out; // 1: the small-call instantiation (residual loads after the rows; bf16 also prefetches its output lines)
    int sf_tiled;     // NVFP4: 1 = block scales in the 128 x 4 tiles block-scaled GEMMs read
    int all_slots;    // ring kernel, residual + bf16, k = 8: the no-per-slot-test instantiation
};

// Sets the calling thread's moe_finalize_rmsnorm_last_error() text.
void set_last_error(const char* fmt, ...);

// mfr_rows.cu: one CTA (or one cluster of CTAs) per token.
bool rows_supported_cpt(int cpt);
cudaError_t rows_prepare(const Launch& l);   // per-kernel attributes (cluster > 8)
// Resident CTAs per SM of the kernel l selects, with slot data in registers or not.
cudaError_t rows_blocks_per_sm(const Launch& l, bool regslots, int* n);
cudaError_t rows_max_active_clusters(const Launch& l, int* n);
cudaError_t rows_launch(const Params& p, const Launch& l, cudaStream_t s);
// An empty kernel with the plan's launch geometry (for the launch floor).
cudaError_t floor_launch(int* status, const Launch& l, cudaStream_t s);
// The plan's launch geometry and protocol plus the call's loads, a cluster
// barrier and/or its stores (MFR_FLOOR_* bits), no arithmetic.
cudaError_t floor_work_launch(const Params& p, const Launch& l, int work, cudaStream_t s);
// One bounded wait that runs out unless `arrive` (tests of the failure path).
cudaError_t wait_selftest_launch(int* status, long long limit, int arrive, cudaStream_t s);

// mfr_expert_norm.cu: each expert row RMS-normalised before the weighted
// sum.  With regslots the one-pass kernel (k <= 8, cpt <= 2; a cluster of
// `cluster` CTAs per token when cluster > 1), else the two-pass kernel (one
// CTA per token).  Launch uses grid_x, block, cluster, cpt, pdl, regslots.
bool expert_norm_one_pass(int k, int cpt);
cudaError_t expert_norm_prepare(const Launch& l);   // checks the form; cluster > 8 attribute
// Resident CTAs per SM of the one-pass or the two-pass kernel for l's cpt and block.
cudaError_t expert_norm_blocks_per_sm(const Launch& l, bool one_pass, int* n);
cudaError_t expert_norm_max_active_clusters(const Launch& l, int* n);
cudaError_t expert_norm_launch(const Params& p, const Launch& l, cudaStream_t s);

// mfr_stream.cu: persistent CTAs fed by bulk copies into a shared-memory ring.
int stream_threads();
int stream_stage_bytes(int k, bool fused);
int stream_smem_bytes(int k, int nstages, bool fused);
cudaError_t stream_prepare(int H, bool fused, bool fp4, int smem_bytes, bool en = false, bool sf_tiled = false,
                           bool all_slots = false);
cudaError_t stream_launch(const Params& p, const Launch& l, cudaStream_t s);

}  // namespace mfr
