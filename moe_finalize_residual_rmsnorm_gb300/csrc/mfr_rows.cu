// Register-gather kernel: one CTA per token (MFR_VARIANT_ROWS), or a
// cluster of C CTAs per token that split the hidden dimension and combine
// their sums of squares through distributed shared memory
// (MFR_VARIANT_CLUSTER).
//
// Per token t, for the columns this CTA owns:
//   trigger   : let the next kernel in the stream start its prologue — at
//               entry when the grid is small (few tokens: its CTAs leave room),
//               else after the loads, so a following kernel does not park CTAs
//               on every SM for the whole call
//   prologue  : slot indices and weights of t (into registers with RS), gamma,
//               (FP4) the encode scale of each of the 256 scale bytes; ask L2
//               to prefetch the CTA's row and residual segments; complete the
//               cluster barrier                             (before the PDL wait)
//   wait      : the producer of expert_out / residual_in has finished
//   gather    : k rows of expert_out, 16 bytes per load, all loads of a slot
//               group issued before any is used
//   accumulate: acc = fma(w_j, e_j, acc) for j = 0..k-1 in slot order
//               (FlashInfer PR 5319 analysis, section 1: FP32 FMA, BF16 at the end)
//   residual  : x = residual_in + acc, written to residual_out
//               (FlashInfer PR 4730 analysis, section 2: sum, residual, RMSNorm fused)
//   reduce    : sum of x^2 — per thread in column order, a warp butterfly,
//               then warps in index order; in a cluster every warp pushes its
//               partial into every CTA's shared memory with st.async, counted
//               on that CTA's mbarrier, and each CTA sums the partials in
//               (rank, warp) order (PR 4730 analysis, section 2: cluster
//               exchange through distributed shared memory)
//   normalise : y = (x * rsqrt(ss / H + eps)) * gamma, rounded to bf16, or
//               (FP4) quantised to NVFP4: 16-element blocks with an E4M3
//               scale, E2M1 codes (PR 6544 analysis, section 2.3: RMSNorm
//               fused with NVFP4 quantisation)
// With FUSED = false the kernel is the plain finalize of the PR 5319 page:
// out = bf16(acc), no residual, no norm; the C CTAs of a token then split
// the columns without a cluster (nothing to reduce).
// Every reduction order is fixed by (H, k, launch geometry), so a plan gives
// bitwise-identical results on every run.
#include <cooperative_groups.h>

#include "mfr_device.cuh"
#include "mfr_internal.h"

namespace cg = cooperative_groups;


namespace mfr {
namespace {

// CPT: 16-byte column chunks per thread per row; SG: slots gathered together;
// FUSED: residual + RMSNorm (true) or plain finalize (false); RS: each
// thread holds the slot rows and weights in registers from before the
// dependency wait (true), or reads them from shared memory as it loads (false:
// 32 fewer registers, for CTAs whose residency the registers would halve);
// PFO: the smallest fused calls (see kPrefetchOutMaxElems; a separate
// instantiation, so larger calls keep the code they were tuned with): the
// residual loads follow the row loads, and the bf16 form also asks L2 for its
// output lines before the wait.
template <int CPT, int SG, bool FUSED, bool FP4, bool RS, bool PFO = false, bool SFT = false>
__global__ void __launch_bounds__(kRowsMaxThreads)
rows_kernel(const Params p, const int csize)
{
    const int tid = threadIdx.x;
    const int nthreads = blockDim.x;
    const int64_t t = blockIdx.x / csize;
    const int rank = static_cast<int>(blockIdx.x - t * csize);
    const int nck = (p.H >> 3) / csize;        // chunks of this CTA
    const int64_t col0 = static_cast<int64_t>(rank) * nck * 8;
    const bool cluster = FUSED && csize > 1;

    __shared__ int s_row[kMaxK];
    __shared__ float s_w[kMaxK];
    __shared__ float s_warp[kRowsMaxThreads / 32];
    __shared__ float s_part[16 * (kRowsMaxThreads / 32)];   // cluster: (rank, warp) partials
    __shared__ float s_enc_tab[FP4 ? 256 : 1];               // FP4: encode scale per scale byte

    if (p.early_trigger)
        pdl_launch_dependents();   // the next kernel may start its prologue now
    // cluster exchange: every CTA will receive one partial sum (4 bytes) from
    // each warp of each CTA of the cluster on s_bar; peers send only after the
    // cluster barrier completes, which also publishes the barrier's
    // initialisation
    __shared__ __align__(8) uint64_t s_bar;
    if (cluster) {
        if (tid == 0) {
            mbar_init(smem_addr(&s_bar), 1);
            mbar_arrive_expect_tx(smem_addr(&s_bar),
                                  static_cast<uint32_t>(csize) * static_cast<uint32_t>(nthreads >> 5) * 4u);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        }
        __syncthreads();
        cg::this_cluster().barrier_arrive();
    }

    // ---- prologue: inputs that the producing kernel does not write --------
    if (tid < p.k) {
        const int32_t r = p.permuted_row_of[t * p.k + tid];
        const bool ok = (r >= 0) && (static_cast<int64_t>(r) < p.R);
        if (!ok && rank == 0 && !(p.sentinel && r < 0))   // negative = non-local when allowed
            atomicOr(p.status, MFR_STATUS_BAD_INDEX);
        s_row[tid] = ok ? r : -1;
        s_w[tid] = p.topk_weights[t * p.k + tid];
    }
    uint4 g[CPT];
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int c = tid + i * nthreads;
        g[i] = (FUSED && c < nck) ? *reinterpret_cast<const uint4*>(p.gamma + col0 + c * 8)
                                  : make_uint4(0, 0, 0, 0);
    }
    if constexpr (FP4) {
        // enc(s8) = 1 / (value(s8) / s_enc), 0 for s8 = 0: the two divisions
        // of each block done once per scale byte, before the wait
        for (int i = tid; i < 256; i += nthreads)
            s_enc_tab[i] = i == 0 ? 0.f : __fdiv_rn(1.0f, __fdiv_rn(e4m3_to_f32(static_cast<uint32_t>(i)), p.s_enc));
    }
    __syncthreads();

    // warm L2 with this CTA's row segments and residual segment while the
    // previous kernel finishes
    if (tid < p.k && s_row[tid] >= 0)
        prefetch_l2_bulk(p.expert_out + static_cast<int64_t>(s_row[tid]) * p.H + col0,
                         static_cast<uint32_t>(nck) * 16u);
    else if (FUSED && tid == kMaxK)
        prefetch_l2_bulk(p.residual_in + t * p.H + col0, static_cast<uint32_t>(nck) * 32u);
    if constexpr (PFO && FUSED && !FP4) {   // the output lines too
        if (tid == kMaxK + 1)
            prefetch_l2_bulk(p.residual_out + t * p.H + col0, static_cast<uint32_t>(nck) * 32u);
        else if (tid == kMaxK + 2)
            prefetch_l2_bulk(p.out + t * p.H + col0, static_cast<uint32_t>(nck) * 16u);
    }

    // RS: slot rows and weights go to registers before the wait, so that
    // after it nothing but address arithmetic stands between the wait and the
    // loads (measured on decode calls: with the shared-memory reads after the
    // wait, the time from the wait to the last row doubled).  Threads past
    // the CTA's chunks load chunk 0 again and discard it, so no load needs a
    // per-thread branch; an invalid slot (-1) is not loaded at all.
    int rr[RS ? kMaxK : 1];
    float ww[RS ? kMaxK : 1];
    if constexpr (RS) {
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) {
            rr[j] = (j < p.k) ? s_row[j] : -1;
            ww[j] = (j < p.k) ? s_w[j] : 0.f;
        }
    }
    auto row_of = [&](int j) -> int {
        if constexpr (RS) return rr[j]; else return (j < p.k) ? s_row[j] : -1;
    };
    auto weight_of = [&](int j) -> float {
        if constexpr (RS) return ww[j]; else return s_w[j];
    };

    // The cluster barrier (arrived at entry) completes here, before the wait,
    // so it costs nothing on the path from the producer to this call's end.
    if (cluster)
        cg::this_cluster().barrier_wait();

    pdl_wait();

    // ---- residual row and the k expert rows ---------------------------------
    // The smallest calls (PFO) issue the residual loads after the first slot
    // group's row loads, so the rows that the first FMAs need come back first
    // (measured: T = 1 / 2 / 4 at H = 4096 3.3 / 3.9 / 3.1 % faster); the same
    // order in the other instantiations made them 11-24 % slower (T = 8 ...
    // 128 at H = 4096 before T = 8 moved to this instantiation), so they load
    // the residual first.
    constexpr bool kResidualAfterRows = PFO;
    float res[CPT][8];
    auto load_residual = [&]() {
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const int c = tid + i * nthreads;
            const int cc = c < nck ? c : 0;
            if (FUSED) {
                const float* res_in = p.residual_in + t * p.H + col0;
                const float4 a = ld_once_f4(res_in + cc * 8);
                const float4 b = ld_once_f4(res_in + cc * 8 + 4);
                res[i][0] = a.x; res[i][1] = a.y; res[i][2] = a.z; res[i][3] = a.w;
                res[i][4] = b.x; res[i][5] = b.y; res[i][6] = b.z; res[i][7] = b.w;
            } else {
#pragma unroll
                for (int q = 0; q < 8; ++q) res[i][q] = 0.f;
            }
        }
    };
    if constexpr (!kResidualAfterRows) load_residual();

    float acc[CPT][8];
#pragma unroll
    for (int i = 0; i < CPT; ++i)
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[i][q] = 0.f;

    // RS: fully unrolled, so rr/ww are indexed by constants and stay in
    // registers; otherwise a plain loop over the slot groups
#pragma unroll
    for (int j0 = 0; j0 < (RS ? kMaxK : p.k); j0 += SG) {
        if (j0 >= p.k) break;
        uint4 v[SG][CPT];
#pragma unroll
        for (int s = 0; s < SG; ++s) {
            const int r = row_of(j0 + s);   // the same for every thread: a uniform branch
            const uint16_t* row = p.expert_out + static_cast<int64_t>(r < 0 ? 0 : r) * p.H + col0;
#pragma unroll
            for (int i = 0; i < CPT; ++i) {
                const int c = tid + i * nthreads;
                v[s][i] = make_uint4(0, 0, 0, 0);
                if (r >= 0) v[s][i] = ld_stream_u4(row + (c < nck ? c : 0) * 8);
            }
        }
        if constexpr (kResidualAfterRows) {
            if (j0 == 0) load_residual();   // after the first group's row loads, before any FMA
        }
#pragma unroll
        for (int s = 0; s < SG; ++s) {
            const int j = j0 + s;
            if (row_of(j) >= 0) {
                const float wj = weight_of(j);
#pragma unroll
                for (int i = 0; i < CPT; ++i) {
                    float e[8];
                    unpack8(v[s][i], e);
#pragma unroll
                    for (int q = 0; q < 8; ++q) acc[i][q] = __fmaf_rn(wj, e[q], acc[i][q]);
                }
            }
        }
    }

    if (!p.early_trigger)
        pdl_launch_dependents();   // every load of this CTA has landed

    if constexpr (!FUSED) {
        // ---- plain finalize: out = bf16(acc) --------------------------------
        uint16_t* out = p.out + t * p.H + col0;
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const int c = tid + i * nthreads;
            if (c < nck) {
                uint4 o;
                o.x = pack_bf16x2(acc[i][0], acc[i][1]);
                o.y = pack_bf16x2(acc[i][2], acc[i][3]);
                o.z = pack_bf16x2(acc[i][4], acc[i][5]);
                o.w = pack_bf16x2(acc[i][6], acc[i][7]);
                st_u4(out + c * 8, o);
            }
        }
        return;
    }

    // ---- x = residual + acc; write the residual; sum of squares ------------
    float* res_out = p.residual_out + t * p.H + col0;
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int c = tid + i * nthreads;
        if (c < nck) {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                acc[i][q] = res[i][q] + acc[i][q];
                ss = __fmaf_rn(acc[i][q], acc[i][q], ss);
            }
            st_f4(res_out + c * 8, make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]));
            st_f4(res_out + c * 8 + 4, make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]));
        }
    }

    ss = warp_allreduce_sum(ss);
    float tot = 0.f;
    const int nwarps = nthreads >> 5;
    if (cluster) {
        // One-way delivery of each warp's partial into slot [rank][warp] of
        // every CTA of the cluster (itself included), lane r writing to CTA r;
        // then wait until all csize * nwarps partials are here and sum them in
        // (rank, warp) order.  No CTA-wide barrier sits on this path (measured:
        // 5-6 % of a decode call).  A CTA leaves only after every write into
        // its shared memory landed.
        const int lane = tid & 31;
        if (lane < csize)
            st_async_cluster_f32(cluster_map(smem_addr(&s_part[rank * nwarps + (tid >> 5)]), lane), ss,
                                 cluster_map(smem_addr(&s_bar), lane));
        if (!mbar_wait(smem_addr(&s_bar), 0))
            atomicOr(p.status, MFR_STATUS_TIMEOUT);
        for (int r = 0; r < csize * nwarps; ++r)
            tot += s_part[r];
    } else {
        if ((tid & 31) == 0)
            s_warp[tid >> 5] = ss;
        __syncthreads();
        for (int w = 0; w < nwarps; ++w)
            tot += s_warp[w];
    }

    // ---- y = (x * inv) * gamma -> bf16 ----------------------------------------
    const float inv = rsqrtf(tot / static_cast<float>(p.H) + p.eps);
    if constexpr (FP4) {
        // NVFP4: chunks c and c^1 (lanes tid and tid^1) form one 16-element block
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const int c = tid + i * nthreads;
            float gf[8], y[8];
            unpack8(g[i], gf);
#pragma unroll
            for (int q = 0; q < 8; ++q) y[q] = (c < nck) ? acc[i][q] * inv * gf[q] : 0.f;
            uint32_t sf;
            const uint32_t w = nvfp4_block8(y, p.s_enc, s_enc_tab, &sf);
            if (c < nck) {
                const int64_t col = col0 + static_cast<int64_t>(c) * 8;
                *reinterpret_cast<uint32_t*>(p.out_q + t * (p.H / 2) + col / 2) = w;
                if ((c & 1) == 0)
                    p.out_sf[nvfp4_sf_index(t, static_cast<int>(col / 16), p.H / 16, SFT)] = static_cast<uint8_t>(sf);
            }
        }
        return;
    }
    uint16_t* out = p.out + t * p.H + col0;
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int c = tid + i * nthreads;
        if (c < nck) {
            float gf[8];
            unpack8(g[i], gf);
            uint4 o;
            o.x = pack_bf16x2(acc[i][0] * inv * gf[0], acc[i][1] * inv * gf[1]);
            o.y = pack_bf16x2(acc[i][2] * inv * gf[2], acc[i][3] * inv * gf[3]);
            o.z = pack_bf16x2(acc[i][4] * inv * gf[4], acc[i][5] * inv * gf[5]);
            o.w = pack_bf16x2(acc[i][6] * inv * gf[6], acc[i][7] * inv * gf[7]);
            st_u4(out + c * 8, o);
        }
    }
}

using RowsKernel = void (*)(const Params, const int);

template <int CPT, int SG, bool RS>
RowsKernel pick_rows(bool fused, bool fp4, bool sft) {
    if (fp4) {
        if (!fused) return nullptr;
        return sft ? rows_kernel<CPT, SG, true, true, RS, false, true> : rows_kernel<CPT, SG, true, true, RS>;
    }
    return fused ? rows_kernel<CPT, SG, true, false, RS> : rows_kernel<CPT, SG, false, false, RS>;
}

// Shared-memory slot reads (RS = false) are instantiated only for one chunk
// per thread: the only case where the registers cost residency (512-thread
// CTAs at 64 vs 112 registers per thread).
RowsKernel rows_kernel_for(int cpt, bool fused, bool fp4, bool regslots, bool pfo = false, bool sft = false) {
    if (pfo) {
        if (cpt != 1 || !fused || !regslots) return nullptr;
        if (fp4) return sft ? rows_kernel<1, 8, true, true, true, true, true> : rows_kernel<1, 8, true, true, true, true>;
        return rows_kernel<1, 8, true, false, true, true>;
    }
    switch (cpt) {
        case 1: return regslots ? pick_rows<1, 8, true>(fused, fp4, sft) : pick_rows<1, 8, false>(fused, fp4, sft);
        case 2: return regslots ? pick_rows<2, 8, true>(fused, fp4, sft) : nullptr;
        case 4: return regslots ? pick_rows<4, 2, true>(fused, fp4, sft) : nullptr;
        default: return nullptr;
    }
}

void fill_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attrs, const Launch& l,
                 cudaStream_t s) {
    cfg = cudaLaunchConfig_t{};
    cfg.gridDim = dim3(static_cast<unsigned>(l.grid_x), static_cast<unsigned>(l.grid_y), 1);
    cfg.blockDim = dim3(static_cast<unsigned>(l.block), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(l.smem_bytes);
    cfg.stream = s;
    int n = 0;
    if (l.cluster > 1 && (l.fused || l.expert_norm)) {   // the plain finalize splits H without a cluster
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

// Same launch protocol as the real kernels and nothing else: the PDL trigger
// and wait.  Timing it with a plan's exact geometry gives the launch floor.
__global__ void floor_kernel(int* status) {
    pdl_launch_dependents();
    pdl_wait();
    if (status == nullptr && threadIdx.x == 0x7FFFFFFF) *status = 0;  // never taken; keeps the argument
}

// The launch-plus-one-pass floor of a fused plan: the plan's exact launch
// geometry and dependent-launch protocol (trigger, cluster barrier arrived at
// entry and completed before the wait, slot indices read and the CTA's row
// and residual segments, and for the smallest calls its output lines,
// prefetched into L2 before the wait), then, by the
// bits of `work`, the call's data movement without its arithmetic:
//   MFR_FLOOR_LOAD      every thread loads its 16-byte chunks of the k slot
//                       rows and of the residual (the call's reads)
//   MFR_FLOOR_EXCHANGE  one cluster-wide barrier (a CTA barrier without a
//                       cluster): the least a cross-CTA reduction can cost
//   MFR_FLOOR_STORE     every thread stores its chunks of residual_out (the
//                       residual it loaded) and out (the XOR of its row
//                       chunks): the call's writes
// Benchmarks time it beside a call to split the call's time into launch,
// data movement, exchange and the kernel's own work.
constexpr int kFloorPrefetchOut = 8;   // internal bit: the plan prefetches its output lines

template <int CPT>
__global__ void __launch_bounds__(kRowsMaxThreads)
floor_work_kernel(const Params p, const int csize, const int work)
{
    const int tid = threadIdx.x;
    const int nthreads = blockDim.x;
    const int64_t t = blockIdx.x / csize;
    const int rank = static_cast<int>(blockIdx.x - t * csize);
    const int nck = (p.H >> 3) / csize;
    const int64_t col0 = static_cast<int64_t>(rank) * nck * 8;
    const bool cluster = csize > 1;
    const bool load = work & MFR_FLOOR_LOAD, store = work & MFR_FLOOR_STORE;
    __shared__ int s_row[kMaxK];

    if (p.early_trigger) pdl_launch_dependents();
    if (cluster) cg::this_cluster().barrier_arrive();
    if (tid < p.k) {
        const int32_t r = p.permuted_row_of[t * p.k + tid];
        s_row[tid] = (r >= 0 && static_cast<int64_t>(r) < p.R) ? r : -1;
    }
    __syncthreads();
    if (load) {
        if (tid < p.k && s_row[tid] >= 0)
            prefetch_l2_bulk(p.expert_out + static_cast<int64_t>(s_row[tid]) * p.H + col0,
                             static_cast<uint32_t>(nck) * 16u);
        else if (tid == kMaxK)
            prefetch_l2_bulk(p.residual_in + t * p.H + col0, static_cast<uint32_t>(nck) * 32u);
    }
    if (store && (work & kFloorPrefetchOut)) {   // as the plan's kernel does for the smallest calls
        if (tid == kMaxK + 1)
            prefetch_l2_bulk(p.residual_out + t * p.H + col0, static_cast<uint32_t>(nck) * 32u);
        else if (tid == kMaxK + 2)
            prefetch_l2_bulk(p.out + t * p.H + col0, static_cast<uint32_t>(nck) * 16u);
    }
    int rr[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) rr[j] = (j < p.k) ? s_row[j] : -1;
    if (cluster) cg::this_cluster().barrier_wait();
    pdl_wait();

    float4 ra[CPT], rb[CPT];
    uint4 fold[CPT];
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        ra[i] = rb[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        fold[i] = make_uint4(0, 0, 0, 0);
    }
    if (load) {
        const float* res_in = p.residual_in + t * p.H + col0;
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const int c = tid + i * nthreads;
            const int cc = c < nck ? c : 0;
            ra[i] = ld_once_f4(res_in + cc * 8);
            rb[i] = ld_once_f4(res_in + cc * 8 + 4);
        }
#pragma unroll
        for (int j = 0; j < kMaxK; ++j) {
            if (rr[j] < 0) continue;   // the same for every thread
            const uint16_t* row = p.expert_out + static_cast<int64_t>(rr[j]) * p.H + col0;
#pragma unroll
            for (int i = 0; i < CPT; ++i) {
                const int c = tid + i * nthreads;
                const uint4 v = ld_stream_u4(row + (c < nck ? c : 0) * 8);
                fold[i].x ^= v.x; fold[i].y ^= v.y; fold[i].z ^= v.z; fold[i].w ^= v.w;
            }
        }
    }
    if (!p.early_trigger) pdl_launch_dependents();
    if (work & MFR_FLOOR_EXCHANGE) {
        if (cluster) cg::this_cluster().sync();
        else __syncthreads();
    }
    if (store) {
        float* res_out = p.residual_out + t * p.H + col0;
        uint16_t* out = p.out + t * p.H + col0;
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const int c = tid + i * nthreads;
            if (c < nck) {
                st_f4(res_out + c * 8, ra[i]);
                st_f4(res_out + c * 8 + 4, rb[i]);
                st_u4(out + c * 8, fold[i]);
            }
        }
    } else if (load && p.T < 0) {
        // never taken (T >= 1 here): keeps the loaded values live without a store
        *p.status = static_cast<int>(fold[0].x ^ __float_as_uint(ra[0].x));
    }
}

// One thread waits, with the kernels' bounded-wait helper, on an mbarrier
// that gets its one arrival only if `arrive`; a wait that runs out sets
// MFR_STATUS_TIMEOUT.  Exercises the failure path without faulting anything.
__global__ void wait_selftest_kernel(int* status, long long limit, int arrive) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(smem_addr(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (arrive) mbar_arrive(smem_addr(&bar));
    if (!mbar_wait_bounded(smem_addr(&bar), 0, limit))
        atomicOr(status, MFR_STATUS_TIMEOUT);
}

}  // namespace

cudaError_t wait_selftest_launch(int* status, long long limit, int arrive, cudaStream_t s) {
    wait_selftest_kernel<<<1, 32, 0, s>>>(status, limit, arrive);
    return cudaGetLastError();
}

cudaError_t floor_launch(int* status, const Launch& l, cudaStream_t s) {
    if (l.smem_bytes > 0) {
        cudaError_t e = cudaFuncSetAttribute(floor_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             l.smem_bytes);
        if (e != cudaSuccess) return e;
    }
    if (l.cluster > 8) {
        cudaError_t e = cudaFuncSetAttribute(floor_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attrs[2];
    fill_config(cfg, attrs, l, s);
    return cudaLaunchKernelEx(&cfg, floor_kernel, status);
}

cudaError_t floor_work_launch(const Params& p, const Launch& l, int work, cudaStream_t s) {
    using K = void (*)(const Params, const int, const int);
    K k = l.cpt == 1 ? floor_work_kernel<1> : l.cpt == 2 ? floor_work_kernel<2> : l.cpt == 4 ? floor_work_kernel<4>
                                                                                            : nullptr;
    if (!k) return cudaErrorInvalidValue;
    if (l.cluster > 8) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attrs[2];
    fill_config(cfg, attrs, l, s);
    return cudaLaunchKernelEx(&cfg, k, p, l.cluster, work | (l.prefetch_out ? kFloorPrefetchOut : 0));
}

bool rows_supported_cpt(int cpt) { return rows_kernel_for(cpt, true, false, true) != nullptr; }

cudaError_t rows_blocks_per_sm(const Launch& l, bool regslots, int* n) {
    RowsKernel k = rows_kernel_for(l.cpt, l.fused != 0, l.fp4 != 0, regslots, false, l.sf_tiled != 0);
    if (!k) { *n = 0; return cudaSuccess; }
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, k, l.block, static_cast<size_t>(l.smem_bytes));
}

cudaError_t rows_prepare(const Launch& l) {
    RowsKernel k = rows_kernel_for(l.cpt, l.fused != 0, l.fp4 != 0, l.regslots != 0, l.prefetch_out != 0,
                                   l.sf_tiled != 0);
    if (!k) return cudaErrorInvalidValue;
    if (l.cluster > 8 && l.fused)
        return cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return cudaSuccess;
}

cudaError_t rows_max_active_clusters(const Launch& l, int* n) {
    RowsKernel k = rows_kernel_for(l.cpt, l.fused != 0, l.fp4 != 0, l.regslots != 0, l.prefetch_out != 0,
                                   l.sf_tiled != 0);
    if (!k) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attrs[2];
    fill_config(cfg, attrs, l, nullptr);
    return cudaOccupancyMaxActiveClusters(n, k, &cfg);
}

cudaError_t rows_launch(const Params& p, const Launch& l, cudaStream_t s) {
    RowsKernel k = rows_kernel_for(l.cpt, l.fused != 0, l.fp4 != 0, l.regslots != 0, l.prefetch_out != 0,
                                   l.sf_tiled != 0);
    if (!k) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attrs[2];
    fill_config(cfg, attrs, l, s);
    return cudaLaunchKernelEx(&cfg, k, p, l.cluster);
}

}  // namespace mfr
