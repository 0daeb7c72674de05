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
// Two kernels; thread tid owns the 16-byte column chunks
// c = tid + i * blockDim.x of every row of its CTA's columns.
//
// expert_norm_reg_kernel (k <= 8, at most two chunks per thread and row):
// one CTA per token, or a cluster of C CTAs per token that split H (small
// calls).  Every row is read once and stays in registers:
//   prologue : slot rows and weights, gamma, an L2 prefetch of the CTA's row
//              segments, the cluster barrier               (before the PDL wait)
//   gather   : the k row segments, all loads issued before any is used
//   sums     : per-slot FP32 sums of squares over the thread's chunks (bf16
//              operands straight into the FMA); per warp a reduce-scatter
//              butterfly; every warp's 8 slot sums go to every CTA of the
//              cluster (st.async into slot [rank][warp][j], counted on that
//              CTA's mbarrier), and lane j of each warp adds slot j over
//              (rank, warp) in order to form c_j
//   sum      : acc = fma(c_j, e_j, acc) in slot order from the registers
//   store    : bf16(gamma * acc)
// expert_norm_kernel (any k <= 16, up to four chunks per thread): one CTA per
// token in two passes; pass 1 forms the per-slot sums of squares (per slot a
// warp butterfly, then the warps in index order), pass 2 reloads the rows (L2 hits, read
// microseconds earlier) for the weighted sum, so no thread holds k rows.
// The ring kernel (mfr_stream.cu, EN) computes the same for large calls with
// k <= 8 and H <= 8192.  HBM sees every row once in all three.  Every order
// is fixed by (H, k, launch geometry), so results are bitwise reproducible.
#include <cooperative_groups.h>

#include "mfr_device.cuh"
#include "mfr_internal.h"

namespace cg = cooperative_groups;

namespace mfr {
namespace {

constexpr int kRegSlots = 8;   // slots the register form holds

template <int CPT>
__global__ void __launch_bounds__(kRowsMaxThreads)
expert_norm_reg_kernel(const Params p, const int csize)
{
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nthreads = blockDim.x;
    const int nwarps = nthreads >> 5;
    const int64_t t = blockIdx.x / csize;
    const int rank = static_cast<int>(blockIdx.x - t * csize);
    const int nck = (p.H >> 3) / csize;        // chunks of this CTA
    const int64_t col0 = static_cast<int64_t>(rank) * nck * 8;
    const bool cluster = csize > 1;

    __shared__ int s_row[kRegSlots];
    __shared__ float s_w[kRegSlots];
    __shared__ float s_part[16 * (kRowsMaxThreads / 32) * kRegSlots];   // [rank][warp][slot]
    __shared__ __align__(8) uint64_t s_bar;

    if (p.early_trigger)
        pdl_launch_dependents();
    // every CTA receives 8 slot sums from each warp of each CTA on s_bar;
    // peers send only after the cluster barrier, which also publishes the
    // barrier's initialisation
    if (cluster) {
        if (tid == 0) {
            mbar_init(smem_addr(&s_bar), 1);
            mbar_arrive_expect_tx(smem_addr(&s_bar),
                                  static_cast<uint32_t>(csize) * static_cast<uint32_t>(nwarps) * kRegSlots * 4u);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        __syncthreads();
        cg::this_cluster().barrier_arrive();
    }

    // ---- prologue: inputs that the producing kernel does not write --------
    if (tid < kRegSlots) {
        int32_t r = -1;
        float w = 0.f;
        if (tid < p.k) {
            r = p.permuted_row_of[t * p.k + tid];
            const bool ok = (r >= 0) && (static_cast<int64_t>(r) < p.R);
            if (!ok && rank == 0 && !(p.sentinel && r < 0))
                atomicOr(p.status, MFR_STATUS_BAD_INDEX);
            r = ok ? r : -1;
            w = p.topk_weights[t * p.k + tid];
        }
        s_row[tid] = r;
        s_w[tid] = w;
    }
    uint4 g[CPT];
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int c = tid + i * nthreads;
        g[i] = c < nck ? *reinterpret_cast<const uint4*>(p.gamma + col0 + c * 8) : make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    if (tid < kRegSlots && s_row[tid] >= 0)
        prefetch_l2_bulk(p.expert_out + static_cast<int64_t>(s_row[tid]) * p.H + col0,
                         static_cast<uint32_t>(nck) * 16u);
    int rr[kRegSlots];
#pragma unroll
    for (int j = 0; j < kRegSlots; ++j) rr[j] = s_row[j];
    if (cluster)
        cg::this_cluster().barrier_wait();

    pdl_wait();

    // ---- gather: every row segment of the CTA, once -------------------------
    uint4 v[kRegSlots][CPT];
#pragma unroll
    for (int j = 0; j < kRegSlots; ++j) {
        const uint16_t* row = p.expert_out + static_cast<int64_t>(rr[j] < 0 ? 0 : rr[j]) * p.H + col0;
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const int c = tid + i * nthreads;
            v[j][i] = make_uint4(0, 0, 0, 0);
            if (rr[j] >= 0) v[j][i] = ld_stream_u4(row + (c < nck ? c : 0) * 8);
        }
    }

    // ---- per-slot sums of squares -> c_j ------------------------------------
    float ss[kRegSlots];
#pragma unroll
    for (int j = 0; j < kRegSlots; ++j) {
        ss[j] = 0.f;
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            if (tid + i * nthreads < nck) {
                ss[j] = sumsq_bf16x4(make_uint2(v[j][i].x, v[j][i].y), ss[j]);
                ss[j] = sumsq_bf16x4(make_uint2(v[j][i].z, v[j][i].w), ss[j]);
            }
        }
    }
    const float part = warp_reduce_scatter8(ss, lane);   // slot lane >> 2 of this warp
    const int slot = lane >> 2;
    if (cluster) {
        // lane 4m + q delivers slot m to CTAs q, q + 4, q + 8, q + 12
        const uint32_t local = smem_addr(&s_part[(rank * nwarps + warp) * kRegSlots + slot]);
        for (int r = lane & 3; r < csize; r += 4)
            st_async_cluster_f32(cluster_map(local, static_cast<uint32_t>(r)), part,
                                 cluster_map(smem_addr(&s_bar), static_cast<uint32_t>(r)));
        if (!mbar_wait(smem_addr(&s_bar), 0))
            atomicOr(p.status, MFR_STATUS_TIMEOUT);
    } else {
        if ((lane & 3) == 0) s_part[warp * kRegSlots + slot] = part;
        __syncthreads();
    }
    float cj = 0.f;
    if (lane < kRegSlots) {
        float tot = 0.f;
        for (int e = 0; e < csize * nwarps; ++e) tot += s_part[e * kRegSlots + lane];
        cj = s_w[lane] * rsqrtf(tot / static_cast<float>(p.H) + p.eps);
    }
    float cr[kRegSlots];
#pragma unroll
    for (int j = 0; j < kRegSlots; ++j) cr[j] = __shfl_sync(0xFFFFFFFFu, cj, j);

    // ---- acc = sum_j c_j * e_j; out = gamma * acc ---------------------------------
    float acc[CPT][8];
#pragma unroll
    for (int i = 0; i < CPT; ++i)
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[i][q] = 0.f;
#pragma unroll
    for (int j = 0; j < kRegSlots; ++j) {
        if (rr[j] >= 0) {
#pragma unroll
            for (int i = 0; i < CPT; ++i) {
                float e[8];
                unpack8(v[j][i], e);
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[i][q] = __fmaf_rn(cr[j], e[q], acc[i][q]);
            }
        }
    }

    if (!p.early_trigger)
        pdl_launch_dependents();   // every load of this CTA has landed

    uint16_t* out = p.out + t * p.H + col0;
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

using TwoPassKernel = void (*)(const Params);
using RegKernel = void (*)(const Params, const int);

TwoPassKernel two_pass_kernel_for(int cpt) {
    switch (cpt) {
        case 1: return expert_norm_kernel<1>;
        case 2: return expert_norm_kernel<2>;
        case 4: return expert_norm_kernel<4>;
        default: return nullptr;
    }
}

RegKernel reg_kernel_for(int cpt) {
    switch (cpt) {
        case 1: return expert_norm_reg_kernel<1>;
        case 2: return expert_norm_reg_kernel<2>;
        default: return nullptr;
    }
}

void fill_en_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attrs, const Launch& l, cudaStream_t s) {
    cfg = cudaLaunchConfig_t{};
    cfg.gridDim = dim3(static_cast<unsigned>(l.grid_x), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(l.block), 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    int n = 0;
    if (l.cluster > 1) {
        attrs[n].id = cudaLaunchAttributeClusterDimension;
        attrs[n].val.clusterDim.x = static_cast<unsigned>(l.cluster);
        attrs[n].val.clusterDim.y = 1;
        attrs[n].val.clusterDim.z = 1;
        ++n;
    }
    if (l.pdl) {
        attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = static_cast<unsigned>(n);
}

}  // namespace

bool expert_norm_one_pass(int k, int cpt) { return k <= kRegSlots && reg_kernel_for(cpt) != nullptr; }

cudaError_t expert_norm_prepare(const Launch& l) {
    if (l.regslots) {
        RegKernel k = reg_kernel_for(l.cpt);
        if (!k) return cudaErrorInvalidValue;
        if (l.cluster > 8) return cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        return cudaSuccess;
    }
    return (l.cluster == 1 && two_pass_kernel_for(l.cpt)) ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t expert_norm_blocks_per_sm(const Launch& l, bool one_pass, int* n) {
    const void* k = one_pass ? reinterpret_cast<const void*>(reg_kernel_for(l.cpt))
                             : reinterpret_cast<const void*>(two_pass_kernel_for(l.cpt));
    if (!k) { *n = 0; return cudaSuccess; }
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, k, l.block, 0);
}

cudaError_t expert_norm_max_active_clusters(const Launch& l, int* n) {
    RegKernel k = reg_kernel_for(l.cpt);
    if (!k || !l.regslots) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attrs[2];
    fill_en_config(cfg, attrs, l, nullptr);
    return cudaOccupancyMaxActiveClusters(n, k, &cfg);
}

cudaError_t expert_norm_launch(const Params& p, const Launch& l, cudaStream_t s) {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attrs[2];
    fill_en_config(cfg, attrs, l, s);
    if (l.regslots) {
        RegKernel k = reg_kernel_for(l.cpt);
        if (!k || p.k > kRegSlots) return cudaErrorInvalidValue;
        return cudaLaunchKernelEx(&cfg, k, p, l.cluster);
    }
    TwoPassKernel k = two_pass_kernel_for(l.cpt);
    if (!k || l.cluster != 1) return cudaErrorInvalidValue;
    return cudaLaunchKernelEx(&cfg, k, p);
}

}  // namespace mfr
