// Finalize with an RMSNorm per expert row before the weighted sum.
//
// The PR 6544 analysis ("FlashInfer, Muse-Spark-Open을 위한 융합 정규화 및
// TP/EP MoE 최적화로 성능 극대화", section 2.1) names a TP MoE finalize that
// fuses the TP reduction, an RMSNorm per expert and the weighted accumulation
// straight from the GEMM2 result, without a formula.  On one GPU the TP
// reduction is the identity; the reading built here normalises every gathered
// expert row over its H columns with the shared gamma and sums the normalised
// rows with the router weights.  In FP32, with the weight folded into the
// row's scale:
//     c_j       = w[t,j] * rsqrt(mean_h(E[r_j, :]^2) + eps)
//     out[t, h] = bf16( gamma[h] * sum_j c_j * E[r_j, h] )
// FMAs in slot order, no residual.
//
// One CTA per token; thread tid owns the 16-byte column chunks
// c = tid + i * blockDim.x of every row.
//   prologue : slot rows into registers, weights to shared memory, gamma, an L2
//              prefetch of the k rows                      (before the PDL wait)
//   pass 1   : the k rows, per-slot FP32 sums of squares over the thread's
//              chunks (fmaf in column order); per slot a warp butterfly and
//              then the warps in index order give c_j
//   pass 2   : the k rows again (L2 hits, read microseconds earlier) and
//              acc = fma(c_j, e, acc) in slot order
//   store    : bf16(gamma * acc)
// The ring kernel (mfr_stream.cu, EN) computes the same for large calls with
// k <= 8 and H <= 8192.
// HBM sees every row once; the second pass trades an L2 round trip for not
// holding k rows per thread in registers.  Every order is fixed by (H, k,
// launch geometry), so results are bitwise reproducible.
#include "mfr_device.cuh"
#include "mfr_internal.h"

namespace mfr {
namespace {

template <int CPT>
__global__ void __launch_bounds__(kRowsMaxThreads)
expert_norm_kernel(const Params p)
{
    constexpr int SG = 8 / CPT;                // slots loaded together (8 chunks of 16 B per thread)
    const int tid = threadIdx.x;
    const int nthreads = blockDim.x;
    const int nwarps = nthreads >> 5;
    const int64_t t = blockIdx.x;
    const int nck = p.H >> 3;                  // 16-byte chunks per row

    __shared__ int s_row[kMaxK];
    __shared__ float s_w[kMaxK];
    __shared__ float s_part[kRowsMaxThreads / 32][kMaxK];
    __shared__ float s_coef[kMaxK];

    if (p.early_trigger)
        pdl_launch_dependents();

    // ---- prologue: inputs that the producing kernel does not write --------
    if (tid < p.k) {
        const int32_t r = p.permuted_row_of[t * p.k + tid];
        const bool ok = (r >= 0) && (static_cast<int64_t>(r) < p.R);
        if (!ok && !(p.sentinel && r < 0))
            atomicOr(p.status, MFR_STATUS_BAD_INDEX);
        s_row[tid] = ok ? r : -1;
        s_w[tid] = p.topk_weights[t * p.k + tid];
    }
    uint4 g[CPT];
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int c = tid + i * nthreads;
        g[i] = c < nck ? *reinterpret_cast<const uint4*>(p.gamma + c * 8) : make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    if (tid < p.k && s_row[tid] >= 0)
        prefetch_l2_bulk(p.expert_out + static_cast<int64_t>(s_row[tid]) * p.H, static_cast<uint32_t>(nck) * 16u);
    int rr[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) rr[j] = (j < p.k) ? s_row[j] : -1;

    pdl_wait();

    // loads slot group [j0, j0 + SG) of this thread's chunks; an invalid
    // slot is not loaded, threads past the row's chunks reload chunk 0
    auto load_group = [&](int j0, uint4 (&v)[SG][CPT]) {
#pragma unroll
        for (int s = 0; s < SG; ++s) {
            const int r = rr[j0 + s];
            const uint16_t* row = p.expert_out + static_cast<int64_t>(r < 0 ? 0 : r) * p.H;
#pragma unroll
            for (int i = 0; i < CPT; ++i) {
                const int c = tid + i * nthreads;
                v[s][i] = make_uint4(0, 0, 0, 0);
                if (r >= 0) v[s][i] = ld_stream_u4(row + (c < nck ? c : 0) * 8);
            }
        }
    };

    // ---- pass 1: per-slot sums of squares -> c_j ------------------------------
#pragma unroll
    for (int j0 = 0; j0 < kMaxK; j0 += SG) {
        if (j0 >= p.k) break;
        uint4 v[SG][CPT];
        load_group(j0, v);
#pragma unroll
        for (int s = 0; s < SG; ++s) {
            float ss = 0.f;
#pragma unroll
            for (int i = 0; i < CPT; ++i) {
                if (tid + i * nthreads < nck) {
                    ss = sumsq_bf16x4(make_uint2(v[s][i].x, v[s][i].y), ss);
                    ss = sumsq_bf16x4(make_uint2(v[s][i].z, v[s][i].w), ss);
                }
            }
            ss = warp_allreduce_sum(ss);
            if ((tid & 31) == 0) s_part[tid >> 5][j0 + s] = ss;
        }
    }
    __syncthreads();
    if (tid < p.k) {
        float tot = 0.f;
        for (int w = 0; w < nwarps; ++w) tot += s_part[w][tid];
        s_coef[tid] = s_w[tid] * rsqrtf(tot / static_cast<float>(p.H) + p.eps);
    }
    __syncthreads();

    // ---- pass 2: acc = sum_j c_j * e_j; out = gamma * acc -----------------------
    float acc[CPT][8];
#pragma unroll
    for (int i = 0; i < CPT; ++i)
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[i][q] = 0.f;
#pragma unroll
    for (int j0 = 0; j0 < kMaxK; j0 += SG) {
        if (j0 >= p.k) break;
        uint4 v[SG][CPT];
        load_group(j0, v);
#pragma unroll
        for (int s = 0; s < SG; ++s) {
            const int j = j0 + s;
            if (rr[j] >= 0) {
                const float cj = s_coef[j];
#pragma unroll
                for (int i = 0; i < CPT; ++i) {
                    float e[8];
                    unpack8(v[s][i], e);
#pragma unroll
                    for (int q = 0; q < 8; ++q) acc[i][q] = __fmaf_rn(cj, e[q], acc[i][q]);
                }
            }
        }
    }

    if (!p.early_trigger)
        pdl_launch_dependents();   // every load of this CTA has landed

    uint16_t* out = p.out + t * p.H;
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int c = tid + i * nthreads;
        if (c < nck) {
            float gf[8];
            unpack8(g[i], gf);
            uint4 o;
            o.x = pack_bf16x2(gf[0] * acc[i][0], gf[1] * acc[i][1]);
            o.y = pack_bf16x2(gf[2] * acc[i][2], gf[3] * acc[i][3]);
            o.z = pack_bf16x2(gf[4] * acc[i][4], gf[5] * acc[i][5]);
            o.w = pack_bf16x2(gf[6] * acc[i][6], gf[7] * acc[i][7]);
            st_u4(out + c * 8, o);
        }
    }
}

using ExpertNormKernel = void (*)(const Params);

ExpertNormKernel expert_norm_kernel_for(int cpt) {
    switch (cpt) {
        case 1: return expert_norm_kernel<1>;
        case 2: return expert_norm_kernel<2>;
        case 4: return expert_norm_kernel<4>;
        default: return nullptr;
    }
}

}  // namespace

cudaError_t expert_norm_launch(const Params& p, const Launch& l, cudaStream_t s) {
    ExpertNormKernel k = expert_norm_kernel_for(l.cpt);
    if (!k) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(l.grid_x), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(l.block), 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attrs[1];
    int n = 0;
    if (l.pdl) {
        attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = static_cast<unsigned>(n);
    return cudaLaunchKernelEx(&cfg, k, p);
}

}  // namespace mfr
