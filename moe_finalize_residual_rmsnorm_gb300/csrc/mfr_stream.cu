// Persistent bulk-copy kernel (MFR_VARIANT_STREAM).
//
// At most one CTA per SM walks a static list of tokens (t = blockIdx.x,
// += gridDim.x); the grid spreads the tokens evenly (stream_grid in mfr_policy.h).
// A producer warp stages, for each token and each column tile of width
// CB = 2048, the k gathered expert-row segments and the residual segment
// into a ring of shared-memory stages with bulk asynchronous copies
// (cp.async.bulk, completion counted in bytes on an mbarrier).  512 consumer
// threads (16 warps, so the schedulers always have a warp whose data is in)
// each own four columns of every tile: they wait for a stage,
// accumulate acc = fma(w_j, e_j, acc) in slot order, add the residual, write
// residual_out, release the stage, and keep x in registers; after the last
// tile of a token they reduce the sum of squares (warp butterfly, then warps
// in index order) and write the bf16 output, or (FP4) its NVFP4 quantisation.
//
// With FUSED = false it is the plain finalize of the PR 5319 page: no
// residual in the stages, out = bf16(acc) written tile by tile, no norm.
//
// With EN = true (FUSED = false, k <= 8, at most 4 tiles) it is the finalize
// with an RMSNorm per expert row, the reading of the PR 6544 analysis, section
// 2.1 (see mfr_expert_norm.cu): each consumer thread keeps its four columns
// of every slot of the first two tiles packed in registers (later tiles stay
// in their ring stages until the second pass) while it sums each slot's
// squares (bf16 operands straight into the FMA), the CTA reduces the k sums
// (a reduce-scatter butterfly in each warp, then thread j adds slot j over
// the warps in index order), c_j = w_j * rsqrt(ss_j / H + eps), and
// out = bf16(gamma * sum_j c_j * e_j) with FMAs in slot order.  The stages
// carry only the rows.
//
// The ring keeps several tiles in flight per SM at all times, so the gather
// never drains between tokens (the register-gather kernel stalls on each
// token's index load and block barrier).  Operation and citations are those
// of the register-gather kernel: FlashInfer PR 5319 analysis section 1 (FP32
// FMA in slot order, bf16 at the end), PR 4730 analysis section 2 (sum,
// residual, RMSNorm fused), PR 5319 analysis section 2 (dependent launch:
// slot indices are read before the wait, rows and residual after it).
//
// Every wait on an mbarrier is bounded: past ~2 s the thread records
// MFR_STATUS_TIMEOUT and stops; before the CTA exits, the producer waits
// (again bounded) for the copies it issued, so no copy is left in flight.
#include "mfr_device.cuh"
#include "mfr_internal.h"

namespace mfr {
namespace {

constexpr int kColsPT = 4;                     // columns per consumer thread and tile
constexpr int kStreamNT = 512;                 // consumer threads (16 warps)
constexpr int kStreamThreads = kStreamNT + 32; // + one producer warp
constexpr int kStreamCB = kStreamNT * kColsPT; // columns per tile (2048)
static_assert(kStreamCB == kStreamTileCols, "the plan policy counts tiles of kStreamTileCols columns");
constexpr int kHeaderBytes = 128;              // per stage: weights + slot mask

struct StageHeader {
    float w[kMaxK];    // at the start of a 128-byte aligned stage: read as float4
    uint32_t mask;
};
static_assert(kMaxK % 4 == 0, "the consumers read the slot weights four at a time");

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return smem_addr(p); }

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global memory into this CTA's shared memory; completion is counted on bar.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// MAXTILES: upper bound on ceil(H / CB) for this instantiation;
// FUSED: residual + RMSNorm (true) or plain finalize (false); EN: per-expert
// RMSNorm (with FUSED = false); SFT (with FP4): block scales in the tiled
// layout of block-scaled GEMMs instead of row-major; AS (residual + bf16 or
// plain finalize, k = 8): tiles whose eight slots are all valid skip the
// per-slot tests (ring_all_slots in mfr_policy.h says where this is taken;
// the per-expert RMSNorm form always has that path).
template <int MAXTILES, bool FUSED, bool FP4, bool EN, bool SFT = false, bool AS = false>
__global__ void __launch_bounds__(kStreamThreads, 1)
stream_kernel(const Params p, const int nstages, const int stage_bytes)
{
    extern __shared__ __align__(128) unsigned char smem[];
    // layout: [nstages full barriers][nstages empty barriers][pad to 128]
    //         then nstages x { header (128 B) | k row segments (CB*2 each) | residual (CB*4) }
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    unsigned char* stages = smem + ((2 * nstages * 8 + 127) / 128) * 128;
    __shared__ float s_warp[kStreamNT / 32];
    __shared__ float s_slot[EN ? kStreamNT / 32 : 1][EN ? 8 : 1];   // EN: per-warp slot sums
    __shared__ float s_coef[EN ? 8 : 1];                            // EN: c_j of the token
    // FP4: the encode scale of every E4M3 block-scale byte for this call's
    // s_enc, enc(s8) = 1 / (value(s8) / s_enc), 0 for s8 = 0, each step the
    // same correctly rounded FP32 operation as per block: two divisions per
    // block become one table read
    __shared__ float s_enc_tab[FP4 ? 256 : 1];
    __shared__ int s_abort;

    const int tid = threadIdx.x;
    const int H = p.H;
    const int k = p.k;
    const int ntiles = (H + kStreamCB - 1) / kStreamCB;
    const int row_bytes = kStreamCB * 2;   // one slot's segment
    const int res_off = kHeaderBytes + k * row_bytes;

    if (tid == 0) {
        for (int s = 0; s < nstages; ++s) {
            mbar_init(smem_u32(&bars[s]), 1);                      // full: producer arrive + tx bytes
            mbar_init(smem_u32(&bars[nstages + s]), kStreamNT / 32); // empty: one arrive per consumer warp
        }
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if constexpr (FP4) {
        for (int i = tid; i < 256; i += blockDim.x)
            s_enc_tab[i] = i == 0 ? 0.f : __fdiv_rn(1.0f, __fdiv_rn(e4m3_to_f32(static_cast<uint32_t>(i)), p.s_enc));
    }
    __syncthreads();

    if (tid >= kStreamNT) {
        // ================= producer warp =================
        // Lane j < k holds slot j of the current token (row index, weight);
        // lane 0 writes the stage header and arms the stage barrier.  The bulk
        // copies of a tile issue either from their own lanes at once (lane j
        // its row, lane kMaxK the residual) or all from lane 0.  Measured on
        // GB300 at the prefill size: issuing from one lane costs ~0.125 us per
        // copy, which caps the plain finalize at 4.8 TB/s (224 us) and parallel
        // issue lifts it to 174 us; the residual + bf16-out form instead runs
        // 6 % faster from one lane (246 vs 263 us, its writes compete with a
        // faster read stream).  The NVFP4 form is 1.4 % faster in parallel at
        // H = 4096 (two tiles per token), but from one lane with four or more
        // tiles (measured: H = 8192 at T = 4096 / 8192 2.8 / 3.5 % faster,
        // T = 16384 with the stress routing 4.3 %, H = 16384 at T = 2048
        // 3.8 %).
        constexpr bool kParallelIssue = !FUSED || (FP4 && MAXTILES <= 2);
        // The residual + bf16 form with four or more tiles per token (H > 4096)
        // issues the first two fills of its ring from the slots' own lanes and
        // the rest from one lane.  Measured on two GB300s against one-lane
        // issue throughout: H = 8192 at T = 1024 / 4096 / 8192 / 32768 1.8 /
        // 2.3 / 2.7 / 2.1 % faster, T = 512 unchanged; at H = 4096 (two tiles)
        // the same change made prefill 1.3 % slower, so those stay one-lane.
        constexpr int64_t kParallelFills = (FUSED && !FP4 && MAXTILES >= 4) ? 2 : 0;
        // No explicit launch_dependents: every CTA of this persistent grid runs
        // from start to end, so an early signal would let a dependent grid park
        // its CTAs on every SM for the whole call (measured: a following
        // producer slowed the pair by 17 %).  Dependents launch as CTAs exit.
        const int lane = tid - kStreamNT;
        int64_t fill = 0;            // stages issued so far
        int s = 0;                   // stage of the next fill
        uint32_t phase = 0;          // how many times the ring wrapped, mod 2
        bool waited = false;
        int64_t t = blockIdx.x;
        // this lane's slot of the first token, loaded ahead
        int32_t nrow = (lane < k && t < p.T) ? p.permuted_row_of[t * k + lane] : -1;
        float nw = (lane < k && t < p.T) ? p.topk_weights[t * k + lane] : 0.f;
        bool ok = true;
        for (; t < p.T && ok; t += gridDim.x) {
            const int32_t row = nrow;
            const float w = nw;
            const int64_t tn = t + gridDim.x;   // load the next token's slot ahead
            nrow = (lane < k && tn < p.T) ? p.permuted_row_of[tn * k + lane] : -1;
            nw = (lane < k && tn < p.T) ? p.topk_weights[tn * k + lane] : 0.f;
            const bool valid = lane < k && row >= 0 && static_cast<int64_t>(row) < p.R;
            const uint32_t mask = __ballot_sync(0xFFFFFFFFu, valid);          // bit j: slot j
            const bool bad = lane < k && !valid && !(p.sentinel && row < 0);  // negative = non-local when allowed
            if (__any_sync(0xFFFFFFFFu, bad) && lane == 0)
                atomicOr(p.status, MFR_STATUS_BAD_INDEX);
            if (!waited) {
                pdl_wait();          // expert_out and residual_in come from the previous kernel
                waited = true;
            }
            for (int b = 0; b < ntiles; ++b) {
                // the consumers released the previous fill of this stage
                const bool freed = fill < nstages || mbar_wait(smem_u32(&bars[nstages + s]), phase ^ 1u);
                if (!__all_sync(0xFFFFFFFFu, freed)) {
                    if (lane == 0) {
                        atomicOr(p.status, MFR_STATUS_TIMEOUT);
                        s_abort = 1;
                    }
                    ok = false;
                    break;
                }
                unsigned char* st = stages + static_cast<size_t>(s) * stage_bytes;
                const int c0 = b * kStreamCB;
                const int cb = min(kStreamCB, H - c0);
                const uint32_t bar = smem_u32(&bars[s]);
                float wl[kMaxK];
#pragma unroll
                for (int j = 0; j < kMaxK; ++j) wl[j] = __shfl_sync(0xFFFFFFFFu, w, j);
                if (lane == 0) {
                    StageHeader* hd = reinterpret_cast<StageHeader*>(st);
#pragma unroll
                    for (int j = 0; j < kMaxK; ++j) hd->w[j] = wl[j];
                    hd->mask = mask;
                    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(__popc(mask) * cb * 2 + (FUSED ? cb * 4 : 0)));
                }
                __syncwarp();
                if (kParallelIssue || (kParallelFills > 0 && fill < kParallelFills)) {
                    if (valid)
                        bulk_g2s(smem_u32(st + kHeaderBytes + lane * row_bytes),
                                 p.expert_out + static_cast<int64_t>(row) * H + c0, static_cast<uint32_t>(cb * 2), bar);
                    if (FUSED && lane == kMaxK)
                        bulk_g2s(smem_u32(st + res_off), p.residual_in + t * H + c0, static_cast<uint32_t>(cb * 4), bar);
                } else {
                    int32_t rl[kMaxK];
#pragma unroll
                    for (int j = 0; j < kMaxK; ++j) rl[j] = __shfl_sync(0xFFFFFFFFu, row, j);
                    if (lane == 0) {
                        // the residual segment first (measured: prefill 246.1 -> 245.3 us)
                        if (FUSED)   // only fused stages carry a residual segment (and count its bytes)
                            bulk_g2s(smem_u32(st + res_off), p.residual_in + t * H + c0, static_cast<uint32_t>(cb * 4), bar);
#pragma unroll
                        for (int j = 0; j < kMaxK; ++j)
                            if (mask & (1u << j))
                                bulk_g2s(smem_u32(st + kHeaderBytes + j * row_bytes),
                                         p.expert_out + static_cast<int64_t>(rl[j]) * H + c0,
                                         static_cast<uint32_t>(cb * 2), bar);
                    }
                }
                ++fill;
                if (++s == nstages) { s = 0; phase ^= 1u; }
            }
        }
        // drain: every copy this warp issued has landed before the CTA exits
        if (lane == 0) {
            for (int64_t f = (fill > nstages ? fill - nstages : 0); f < fill; ++f) {
                const int sf = static_cast<int>(f % nstages);
                if (!mbar_wait(smem_u32(&bars[sf]), static_cast<uint32_t>(f / nstages) & 1u)) {
                    atomicOr(p.status, MFR_STATUS_TIMEOUT);
                    break;
                }
            }
        }
        return;
    }

    // ===================== consumer threads =====================
    // Thread tid owns columns [c0 + 4*tid, c0 + 4*tid + 4) of every tile.
    const int warp = tid >> 5;
    uint32_t g[MAXTILES][2];
#pragma unroll
    for (int b = 0; b < MAXTILES; ++b) {
        const int col = b * kStreamCB + tid * kColsPT;
        uint2 v = make_uint2(0, 0);
        if ((FUSED || EN) && b < ntiles && col < H) v = *reinterpret_cast<const uint2*>(p.gamma + col);
        g[b][0] = v.x; g[b][1] = v.y;
    }
    pdl_wait();

    int s = 0;
    uint32_t phase = 0;
    if constexpr (EN) {
        // ---- RMSNorm per expert row: the rows stay available until the token's c_j are known.
        // A thread keeps its share of the first kRegTiles tiles packed in
        // registers (32 registers) and releases those stages at once; the
        // stages of later tiles (H > 4096) are held until the second pass
        // re-reads them, and the producer refills the stages left over.  At
        // most MAXTILES - kRegTiles = 2 stages are held, so a ring of 2 stages
        // never deadlocks.  Measured at H = 8192, T = 4096: 91.4 us, against
        // 99.1 us holding all four stages (and slower still with all four
        // tiles in 64 registers).
        constexpr int kRegTiles = 2;
        const int lane = tid & 31;
        for (int64_t t = blockIdx.x; t < p.T; t += gridDim.x) {
            uint2 rv[kRegTiles][8];
            float ss[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) ss[j] = 0.f;
            uint32_t mask = 0;
            float my_w = 0.f;       // thread j < 8: the weight of slot j
            bool ok = true;
            const int s0 = s;
            const uint32_t phase0 = phase;
#pragma unroll
            for (int b = 0; b < MAXTILES; ++b) {
                if (b >= ntiles) break;
                const uint32_t bar = smem_u32(&bars[s]);
                const uint32_t ebar = smem_u32(&bars[nstages + s]);
                const unsigned char* st = stages + static_cast<size_t>(s) * stage_bytes;
                const bool landed = __all_sync(0xFFFFFFFFu, mbar_wait(bar, phase));
                if (++s == nstages) { s = 0; phase ^= 1u; }
                if (!landed) {
                    atomicOr(p.status, MFR_STATUS_TIMEOUT);
                    ok = false;
                    break;
                }
                const StageHeader* hd = reinterpret_cast<const StageHeader*>(st);
                mask = hd->mask;
                if (tid < 8) my_w = hd->w[tid];
                const int c0 = b * kStreamCB;
                const bool mine = tid * kColsPT < min(kStreamCB, H - c0);
                const bool in_regs = b < kRegTiles;       // a constant: the loop is unrolled
                const int rb = in_regs ? b : 0;
                if (k == 8 && mask == 0xFFu && mine) {
                    // all eight slots valid: the eight loads first, then the
                    // sums of squares, with no per-slot tests (measured on
                    // GB300: 0.3-4.0 % faster at every size from T = 512 to
                    // 16384, H = 4096 and 8192; prefill 181.7 -> 174.5 us)
                    uint2 vv[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        vv[j] = *reinterpret_cast<const uint2*>(st + kHeaderBytes + j * row_bytes + tid * 8);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (in_regs) rv[rb][j] = vv[j];
                        ss[j] = sumsq_bf16x4(vv[j], ss[j]);   // bf16 operands straight into the FMA
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (in_regs) rv[rb][j] = make_uint2(0, 0);
                        if (j < k && (mask & (1u << j)) && mine) {
                            const uint2 v = *reinterpret_cast<const uint2*>(st + kHeaderBytes + j * row_bytes + tid * 8);
                            if (in_regs) rv[rb][j] = v;
                            ss[j] = sumsq_bf16x4(v, ss[j]);
                        }
                    }
                }
                if (in_regs) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(ebar);     // this warp is done with the stage
                }
            }
            // Per-slot sums over the CTA in a fixed order: the warp's sums by
            // a reduce-scatter butterfly (slot m in lanes 4m..4m+3), then
            // thread j < k adds slot j over the warps in index order.
            {
                const float c = warp_reduce_scatter8(ss, lane);
                if ((lane & 3) == 0) s_slot[warp][lane >> 2] = c;
            }
            const uint32_t stop_in = (!ok || s_abort != 0) ? 1u : 0u;
            uint32_t stop;
            asm volatile("{\n\t.reg .pred pin, pout;\n\t"
                         "setp.ne.u32 pin, %1, 0;\n\t"
                         "bar.red.or.pred pout, 1, %2, pin;\n\t"
                         "selp.u32 %0, 1, 0, pout;\n\t}"
                         : "=r"(stop) : "r"(stop_in), "r"(kStreamNT) : "memory");
            if (stop) break;
            if (tid < k) {
                float tot = 0.f;
#pragma unroll
                for (int w = 0; w < kStreamNT / 32; ++w) tot += s_slot[w][tid];
                s_coef[tid] = my_w * rsqrtf(tot / static_cast<float>(H) + p.eps);
            }
            asm volatile("bar.sync 1, %0;" :: "r"(kStreamNT) : "memory");   // s_coef ready, s_slot reusable
            float cr[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) cr[j] = (j < k) ? s_coef[j] : 0.f;
            int s2 = s0;
            uint32_t phase2 = phase0;
#pragma unroll
            for (int b = 0; b < MAXTILES; ++b) {
                if (b >= ntiles) break;
                const int col = b * kStreamCB + tid * kColsPT;
                const unsigned char* st = stages + static_cast<size_t>(s2) * stage_bytes;
                const uint32_t ebar = smem_u32(&bars[nstages + s2]);
                if (++s2 == nstages) { s2 = 0; phase2 ^= 1u; }
                const bool in_regs = b < kRegTiles;
                const int rb = in_regs ? b : 0;
                float acc[kColsPT];
#pragma unroll
                for (int q = 0; q < kColsPT; ++q) acc[q] = 0.f;
                if (col < H) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (j < k && (mask & (1u << j))) {
                            uint2 v;
                            if (in_regs) v = rv[rb][j];
                            else v = *reinterpret_cast<const uint2*>(st + kHeaderBytes + j * row_bytes + tid * 8);
                            const float e[4] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y)};
#pragma unroll
                            for (int q = 0; q < kColsPT; ++q) acc[q] = __fmaf_rn(cr[j], e[q], acc[q]);
                        }
                    }
                }
                if (!in_regs) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(ebar);     // both passes are done with the stage
                }
                if (col < H) {
                    float y[kColsPT];
#pragma unroll
                    for (int q = 0; q < kColsPT; ++q) {
                        const uint32_t gw = g[b][q >> 1];
                        y[q] = acc[q] * ((q & 1) ? bf16_hi(gw) : bf16_lo(gw));
                    }
                    st_u2(p.out + t * H + col, make_uint2(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3])));
                }
            }
            (void)phase2;
        }
    } else if constexpr (!FUSED) {
        // ---- plain finalize: every tile goes straight to out ----------------
        for (int64_t t = blockIdx.x; t < p.T; t += gridDim.x) {
            bool ok = true;
            for (int b = 0; b < ntiles; ++b) {
                const uint32_t bar = smem_u32(&bars[s]);
                const uint32_t ebar = smem_u32(&bars[nstages + s]);
                const unsigned char* st = stages + static_cast<size_t>(s) * stage_bytes;
                const bool landed = __all_sync(0xFFFFFFFFu, mbar_wait(bar, phase));
                if (++s == nstages) { s = 0; phase ^= 1u; }
                if (!landed) {
                    atomicOr(p.status, MFR_STATUS_TIMEOUT);
                    ok = false;
                    break;
                }
                const StageHeader* hd = reinterpret_cast<const StageHeader*>(st);
                const uint32_t mask = hd->mask;
                const int c0 = b * kStreamCB;
                const bool mine = tid * kColsPT < min(kStreamCB, H - c0);
                float acc[kColsPT];
#pragma unroll
                for (int q = 0; q < kColsPT; ++q) acc[q] = 0.f;
                if (mine && AS && k == 8 && mask == 0xFFu) {
                    // AS: all eight slots valid: loads first, FMAs without per-slot tests
                    uint2 v[8];
                    float wv[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        v[j] = *reinterpret_cast<const uint2*>(st + kHeaderBytes + j * row_bytes + tid * 8);
                        wv[j] = hd->w[j];
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float e[4] = {bf16_lo(v[j].x), bf16_hi(v[j].x), bf16_lo(v[j].y), bf16_hi(v[j].y)};
#pragma unroll
                        for (int q = 0; q < kColsPT; ++q) acc[q] = __fmaf_rn(wv[j], e[q], acc[q]);
                    }
                } else if (mine) {
#pragma unroll
                    for (int j = 0; j < kMaxK; ++j) {
                        if (j < k && (mask & (1u << j))) {
                            const float wj = hd->w[j];
                            const uint2 v = *reinterpret_cast<const uint2*>(st + kHeaderBytes + j * row_bytes + tid * 8);
                            const float e[4] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y)};
#pragma unroll
                            for (int q = 0; q < kColsPT; ++q) acc[q] = __fmaf_rn(wj, e[q], acc[q]);
                        }
                    }
                }
                __syncwarp();
                if ((tid & 31) == 0) mbar_arrive(ebar);
                if (mine)
                    st_u2(p.out + t * H + c0 + tid * kColsPT,
                          make_uint2(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3])));
            }
            if (!ok) break;     // warp-uniform: this warp stops; the others time out on their own
        }
    } else {
    for (int64_t t = blockIdx.x; t < p.T; t += gridDim.x) {
        float x[MAXTILES][kColsPT];
        float ss = 0.f;
        bool ok = true;
#pragma unroll
        for (int b = 0; b < MAXTILES; ++b) {
            if (b >= ntiles) break;
            const uint32_t bar = smem_u32(&bars[s]);
            const uint32_t ebar = smem_u32(&bars[nstages + s]);
            const unsigned char* st = stages + static_cast<size_t>(s) * stage_bytes;
            // one decision per warp, so every lane reaches the same __syncwarp
            const bool landed = __all_sync(0xFFFFFFFFu, mbar_wait(bar, phase));
            if (++s == nstages) { s = 0; phase ^= 1u; }
            if (!landed) {
                atomicOr(p.status, MFR_STATUS_TIMEOUT);
                ok = false;
                break;
            }
            const StageHeader* hd = reinterpret_cast<const StageHeader*>(st);
            const uint32_t mask = hd->mask;
            const int c0 = b * kStreamCB;
            const int cb = min(kStreamCB, H - c0);
            const bool mine = tid * kColsPT < cb;
            float acc[kColsPT];
#pragma unroll
            for (int q = 0; q < kColsPT; ++q) acc[q] = 0.f;
            if (mine) {
                // AS: k = 8 and every slot valid (a uniform test per tile): the
                // eight slots' loads first, then the FMAs, with no per-slot
                // tests (the NVFP4 form was 1-2 % slower with it)
                if (AS && k == 8 && mask == 0xFFu) {
                    uint2 v[8];
                    float wv[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        v[j] = *reinterpret_cast<const uint2*>(st + kHeaderBytes + j * row_bytes + tid * 8);
                        wv[j] = hd->w[j];
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float e[4] = {bf16_lo(v[j].x), bf16_hi(v[j].x), bf16_lo(v[j].y), bf16_hi(v[j].y)};
#pragma unroll
                        for (int q = 0; q < kColsPT; ++q) acc[q] = __fmaf_rn(wv[j], e[q], acc[q]);
                    }
                } else {
                    // up to 8192 columns the slot weights come in four 16-byte
                    // reads of the stage header (measured: prefill 243.9 ->
                    // 242.9 us, stress and wide T = 8192 0.9 / 0.7 % faster
                    // than one read per slot); wider rows keep one read per
                    // slot (the 16 registers would spill there)
                    constexpr bool kWeights4 = MAXTILES <= 4;
                    float wall[kWeights4 ? kMaxK : 1];
                    if constexpr (kWeights4) {
#pragma unroll
                        for (int j4 = 0; j4 < kMaxK; j4 += 4) {
                            const float4 w4 = *reinterpret_cast<const float4*>(&hd->w[j4]);
                            wall[j4] = w4.x; wall[j4 + 1] = w4.y; wall[j4 + 2] = w4.z; wall[j4 + 3] = w4.w;
                        }
                    }
                    // NVFP4: the mask alone decides (the producer sets no
                    // bit at or above k), measured 1.8 / 2.5 % faster at
                    // prefill with row-major / tiled scales and 0.5-1 % at
                    // wide T = 8192 and stress; the bf16 form was 0.1-0.8 %
                    // slower without the slot-count test and keeps it
#pragma unroll
                    for (int j = 0; j < kMaxK; ++j) {
                        if ((FP4 || j < k) && (mask & (1u << j))) {
                            float wj;
                            if constexpr (kWeights4) wj = wall[j]; else wj = hd->w[j];
                            const uint2 v = *reinterpret_cast<const uint2*>(st + kHeaderBytes + j * row_bytes + tid * 8);
                            const float e[4] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y)};
#pragma unroll
                            for (int q = 0; q < kColsPT; ++q) acc[q] = __fmaf_rn(wj, e[q], acc[q]);
                        }
                    }
                }
                const float4 r = *reinterpret_cast<const float4*>(st + res_off + tid * 16);
                x[b][0] = r.x + acc[0]; x[b][1] = r.y + acc[1];
                x[b][2] = r.z + acc[2]; x[b][3] = r.w + acc[3];
            } else {
#pragma unroll
                for (int q = 0; q < kColsPT; ++q) x[b][q] = 0.f;
            }
            __syncwarp();
            if ((tid & 31) == 0) mbar_arrive(ebar);   // this warp is done with the stage
            if (mine) {
#pragma unroll
                for (int q = 0; q < kColsPT; ++q) ss = __fmaf_rn(x[b][q], x[b][q], ss);
                st_f4(p.residual_out + t * H + c0 + tid * kColsPT, make_float4(x[b][0], x[b][1], x[b][2], x[b][3]));
            }
        }
        ss = warp_allreduce_sum(ss);
        if ((tid & 31) == 0) s_warp[warp] = ss;
        // consumer-only barrier that also ORs "stop" over every consumer
        // thread, so all of them take the same decision
        const uint32_t stop_in = (!ok || s_abort != 0) ? 1u : 0u;
        uint32_t stop;
        asm volatile("{\n\t.reg .pred pin, pout;\n\t"
                     "setp.ne.u32 pin, %1, 0;\n\t"
                     "bar.red.or.pred pout, 1, %2, pin;\n\t"
                     "selp.u32 %0, 1, 0, pout;\n\t}"
                     : "=r"(stop) : "r"(stop_in), "r"(kStreamNT) : "memory");
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < kStreamNT / 32; ++w) tot += s_warp[w];
        asm volatile("bar.sync 1, %0;" :: "r"(kStreamNT) : "memory");  // s_warp reusable
        if (stop) break;
        const float inv = rsqrtf(tot / static_cast<float>(H) + p.eps);
#pragma unroll
        for (int b = 0; b < MAXTILES; ++b) {
            if (b >= ntiles) break;
            const int col = b * kStreamCB + tid * kColsPT;
            float y[4];
#pragma unroll
            for (int q = 0; q < kColsPT; ++q) {
                const uint32_t gw = g[b][q >> 1];
                y[q] = x[b][q] * inv * ((q & 1) ? bf16_hi(gw) : bf16_lo(gw));
            }
            if constexpr (FP4) {
                // NVFP4: the four lanes 4m..4m+3 hold one 16-column block
#pragma unroll
                for (int q = 0; q < kColsPT; ++q) if (col >= H) y[q] = 0.f;
                uint32_t sf;
                const uint32_t w = nvfp4_block4(y, p.s_enc, s_enc_tab, &sf);
                if (col < H) {
                    *reinterpret_cast<uint16_t*>(p.out_q + t * (H / 2) + col / 2) = static_cast<uint16_t>(w);
                    if ((tid & 3) == 0)
                        p.out_sf[nvfp4_sf_index(t, col / 16, H / 16, SFT)] = static_cast<uint8_t>(sf);
                }
            } else if (col < H) {
                st_u2(p.out + t * H + col, make_uint2(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3])));
            }
        }
    }
    }  // FUSED
}

using StreamKernel = void (*)(const Params, const int, const int);

template <int MAXTILES>
StreamKernel pick(bool fused, bool fp4, bool sft, bool as) {
    if (fp4) {
        if (!fused) return nullptr;
        return sft ? stream_kernel<MAXTILES, true, true, false, true> : stream_kernel<MAXTILES, true, true, false>;
    }
    if constexpr (MAXTILES <= 4) {
        if (as) return fused ? stream_kernel<MAXTILES, true, false, false, false, true>
                             : stream_kernel<MAXTILES, false, false, false, false, true>;
    }
    if (as) return nullptr;   // not taken above 8192 columns
    return fused ? stream_kernel<MAXTILES, true, false, false> : stream_kernel<MAXTILES, false, false, false>;
}

StreamKernel stream_kernel_for(int H, bool fused, bool fp4, bool en, bool sft = false, bool as = false) {
    const int tiles = (H + kStreamCB - 1) / kStreamCB;
    if (en) {
        if (fused || fp4) return nullptr;
        if (tiles <= 2) return stream_kernel<2, false, false, true>;
        if (tiles <= 4) return stream_kernel<4, false, false, true>;
        return nullptr;
    }
    if (tiles <= 2) return pick<2>(fused, fp4, sft, as);
    if (tiles <= 4) return pick<4>(fused, fp4, sft, as);
    if (tiles <= 8) return pick<8>(fused, fp4, sft, as);
    return nullptr;
}

}  // namespace

int stream_threads() { return kStreamThreads; }

int stream_stage_bytes(int k, bool fused) {
    return kHeaderBytes + k * kStreamCB * 2 + (fused ? kStreamCB * 4 : 0);
}

int stream_smem_bytes(int k, int nstages, bool fused) {
    return ((2 * nstages * 8 + 127) / 128) * 128 + nstages * stream_stage_bytes(k, fused);
}

cudaError_t stream_prepare(int H, bool fused, bool fp4, int smem_bytes, bool en, bool sf_tiled, bool all_slots) {
    StreamKernel kf = stream_kernel_for(H, fused, fp4, en, sf_tiled, all_slots);
    if (!kf) return cudaErrorInvalidValue;
    return cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
}

cudaError_t stream_launch(const Params& p, const Launch& l, cudaStream_t s) {
    StreamKernel kf = stream_kernel_for(p.H, l.fused != 0, l.fp4 != 0, l.expert_norm != 0, l.sf_tiled != 0,
                                        l.all_slots != 0);
    if (!kf) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(l.grid_x), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(l.block), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(l.smem_bytes);
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
    return cudaLaunchKernelEx(&cfg, kf, p, l.stages, stream_stage_bytes(p.k, l.fused != 0));
}

}  // namespace mfr
