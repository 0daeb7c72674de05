// Launch policy of a plan: which kernel, how many CTAs per token, threads and
// grid, from (T, H, k, the plan kind, the options, the ring depth the device
// allows and its SM count).  Pure host code with no CUDA dependency, so the
// CPU tests compile and check it directly; mfr_api.cu applies it.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cstdio>

#include "moe_finalize_rmsnorm.h"

namespace mfr {

constexpr int kMaxK = 16;               // slots per token
constexpr int kMaxH = 16384;            // hidden size
constexpr int kRowsMaxThreads = 512;    // one-CTA-per-token kernels
constexpr int kStreamTileCols = 2048;   // ring kernel: columns per tile
constexpr int kMaxStages = 8;           // ring kernel: deepest ring

// Variant choice by the number of elements T*H of a call (measured on GB300
// with cold inputs, CUDA graph): up to 2^19 a cluster of CTAs per token is
// fastest (few tokens, latency bound; decode_cluster, finalize_split and
// en_cluster pick its size per plan kind); above that one CTA per token
// while its grid is one wave, 8192 elements per SM (304 tokens at H = 4096,
// two CTAs per SM; 152 at H = 8192), and the persistent ring kernel from
// there.  Measured with the ring's all-slots form, forced variants: at the
// wave boundary one CTA per token is 2-19 % faster for every output; one
// wave above it (T = 320 / 352 at H = 4096, 160 / 176 at H = 8192) the ring
// is faster for the residual + bf16 (0.4-6.5 %), plain finalize (2-7.5 %)
// and per-expert RMSNorm (6-16 %) outputs, but 4-6.5 % slower for NVFP4,
// which keeps one CTA per token below 1.5*2^20 (there the ring was 8 %
// faster at H = 4096 and 3 % slower at H = 8192, at 2^21 faster at both).
// Small grids signal their dependents at entry.
constexpr int64_t kClusterMaxElems = int64_t(1) << 19;
constexpr int64_t kRowsMaxElems = int64_t(3) << 19;      // NVFP4: ring from here
constexpr int64_t kRowsElemsPerSm = 8192;                // other outputs: one wave of rows CTAs
inline bool rows_beats_ring(int64_t elems, bool fp4, int sms) {
    return fp4 ? elems < kRowsMaxElems : elems <= kRowsElemsPerSm * sms;
}
constexpr int64_t kEarlyTriggerMaxElems = int64_t(1) << 19;
// Calls this small leave HBM idle, so the fused bf16 kernel also asks L2 for
// its output lines before the dependency wait, so the stores at the end hit,
// and issues its residual loads after its row loads (the rows the first FMAs
// need come back first).  Measured on GB300: T = 1 / 2 / 4 at H = 4096
// 3.3-3.9 % faster with the load order, and with the limit at 2^15 rather
// than 2^14 T = 8 at H = 4096 1.1 % and T = 4 at H = 8192 2.1 % faster,
// 2^16 no different at T = 16.  The output prefetch alone had been 1-4 %
// slower from 2^15 elements on.  The NVFP4 kernel takes the load order but
// not the output prefetch (T = 1 / 2 / 4 / 8 at H = 4096 1.4 / 1.7 / 1.1 /
// 0.7 % faster); the plain finalize and per-expert RMSNorm kernels take
// neither: with the output prefetch they ran 0-8 % slower at the same
// sizes.  It is a separate instantiation, because merely
// adding the branch changed the other instantiations' code (T = 8, H = 4096:
// 1.81 -> 1.84 us without the prefetch taken).
constexpr int64_t kPrefetchOutMaxElems = int64_t(1) << 15;

// The ring kernel's residual + bf16 and plain finalize forms with k = 8
// have an instantiation whose consumers, when all eight slots of a tile are
// valid, load the eight row segments first and then run the FMAs with no
// per-slot tests.  Measured on GB300 against the general slot loop (same
// box, two rounds, outputs hashed equal):
//  residual + bf16: H = 4096, T = 512 / 1024 / 2048 / 4096 2.9 / 3.5 / 2.6 /
//    0.9 % faster; H = 8192, T = 256 / 512 / 1024 / 2048 6.3 / 2.6 / 1.7 /
//    1.4 % faster; prefill (T = 16384, H = 4096) within 0.3 % either way;
//    H = 8192, T = 4096 / 8192 / 32768 0.7 / 1.8 / 1.5 % slower;
//  plain finalize: H = 4096, T = 1024 / 4096 / 16384 11 / 4.5 / 1.0 %
//    faster; H = 8192, T = 512 17 % faster, T = 2048 / 4096 / 8192 0.5 /
//    1.9 / 3.8 % slower.
// So: residual + bf16 up to 2^24 elements at H <= 8192; plain finalize at
// every size up to H = 4096 and up to 2^22 elements at H = 8192.  (The
// per-expert RMSNorm form has the same path in its only instantiation.)
constexpr int64_t kRingAllSlotsMaxElems = int64_t(1) << 24;
constexpr int64_t kPlainAllSlotsMaxElems = int64_t(1) << 22;
inline bool ring_all_slots(int64_t T, int64_t H, int k, bool fused, bool fp4, bool expert_norm) {
    if (fp4 || expert_norm || k != 8 || H > 4 * kStreamTileCols) return false;
    if (fused) return T * H <= kRingAllSlotsMaxElems;
    return H <= 2 * kStreamTileCols || T * H <= kPlainAllSlotsMaxElems;
}

inline int round_up(int v, int m) { return (v + m - 1) / m * m; }

inline int stream_tiles(int H) { return (H + kStreamTileCols - 1) / kStreamTileCols; }

// Smallest chunks-per-thread that keeps a CTA within kRowsMaxThreads threads.
inline int pick_cpt(int chunks) {
    for (int cpt = 1; cpt <= 4; cpt *= 2)
        if ((chunks + cpt - 1) / cpt <= kRowsMaxThreads) return cpt;
    return 0;
}

// Cluster size for the split-H variant: the largest power of two <= cmax
// that divides the chunk count and leaves at least one warp of chunks per CTA.
inline int auto_cluster(int chunks, int cmax = 8) {
    int c = cmax;
    while (c > 1 && (chunks % c != 0 || chunks / c < 32)) c /= 2;
    return c;
}

// The most CTAs per token (a power of two, at most 16) that split the
// chunks evenly and leave each CTA at least `threads` of them.
inline int split_for_threads(int chunks, int threads) {
    int c = 1;
    while (c < 16 && chunks / (2 * c) >= threads && chunks % (2 * c) == 0) c *= 2;
    return c;
}

// Cluster size for a latency-bound call of T*H = elems (measured on GB300, a
// CUDA graph of back-to-back calls, cold inputs, H = 4096 and 8192): up to
// 2^14 elements the fewest CTAs that give each 128 threads (one 16-byte chunk
// per thread: H=4096 -> 4, H=8192 -> 8; 3 % faster than 8 at H=4096, T=1);
// up to 2^17 clusters of 16 (4-9 % faster than 8 at T = 4..32, H = 4096 and
// T = 4..16, H = 8192); up to 2^18, 8 (16 is 7 % slower at T=32, H=8192); up
// to 2^19 the fewest CTAs of 256 threads each (H=4096 -> 2, H=8192 -> 4: 3-5 %
// faster than one CTA per token at H=4096, 9-18 % at H=8192).  1 = no cluster.
inline int decode_cluster(int chunks, int64_t elems) {
    if (elems <= (int64_t(1) << 14)) return split_for_threads(chunks, 128);
    if (elems <= (int64_t(1) << 17)) return auto_cluster(chunks, 16);
    if (elems <= (int64_t(1) << 18)) return auto_cluster(chunks);
    return split_for_threads(chunks, 256);
}

// CTAs per token for a small plain finalize (no residual, no norm: the CTAs
// of a token share nothing, no cluster launch), measured the same way (two
// repetitions within 3 %): CTAs of 64 threads up to 2^13 elements, 32 up to
// 2^14, 256 up to 2^16, 128 up to 2^19.  Against the fused kernel's sizes:
// T = 8 at H = 4096 1.84 -> 1.60 us, T = 4 at H = 8192 1.82 -> 1.59 us.
inline int finalize_split(int chunks, int64_t elems) {
    if (elems <= (int64_t(1) << 13)) return split_for_threads(chunks, 64);
    if (elems <= (int64_t(1) << 14)) return split_for_threads(chunks, 32);
    if (elems <= (int64_t(1) << 16)) return split_for_threads(chunks, 256);
    return split_for_threads(chunks, 128);
}

// Cluster size for a small call of the per-expert RMSNorm form (measured on
// GB300 as decode_cluster was, T = 1..128 at H = 4096 and 8192, two
// repetitions within 0.5 %): up to 2^13 elements CTAs of 128 threads, up to
// 2^15 CTAs of 32 (16 CTAs per token: T = 4 at H = 4096 1.88 us against 2.02
// with 128-thread CTAs), up to 2^16 CTAs of 64 (c16 at H = 8192, T = 8; c8
// at H = 4096, T = 16: 10 % faster than 16), up to 2^18 CTAs of 512 threads
// (one CTA per token at H = 4096, two at 8192: 7-17 % faster than the fused
// kernel's sizes), beyond that one CTA per token.  Its exchange carries 8
// sums per warp, so fewer, larger CTAs win earlier than in the fused kernel.
inline int en_cluster(int chunks, int64_t elems) {
    if (elems <= (int64_t(1) << 13)) return split_for_threads(chunks, 128);
    if (elems <= (int64_t(1) << 15)) return split_for_threads(chunks, 32);
    if (elems <= (int64_t(1) << 16)) return split_for_threads(chunks, 64);
    if (elems <= (int64_t(1) << 18)) return split_for_threads(chunks, 512);
    return 1;
}

// Persistent CTAs for T tokens on `sms` SMs: the fewest rounds of one token
// per CTA, over as few CTAs as give every CTA the same number of tokens (+-1).
// T = 512 on 152 SMs: 128 CTAs x 4 tokens instead of 56 CTAs with 4 and 96
// with 3 (measured 4 % faster at H = 8192, and never slower from T = 200 to
// T = 16384: the last round no longer runs on a fraction of the SMs).
inline int stream_grid(int64_t T, int sms) {
    if (T <= sms) return static_cast<int>(T > 0 ? T : 1);
    const int64_t rounds = (T + sms - 1) / sms;
    return static_cast<int>((T + rounds - 1) / rounds);
}

struct PolicyIn {
    int64_t T, H;
    int k;
    bool fused;          // residual + RMSNorm
    bool fp4;            // NVFP4 output
    bool expert_norm;    // RMSNorm per expert row
    int force_variant;   // MFR_VARIANT_*
    int cluster_size;    // 0 = auto
    int stages;          // ring depth the device's shared memory allows for this plan
    int sms;
};

struct PolicyOut {
    int variant;         // MFR_VARIANT_CLUSTER / _ROWS / _STREAM
    int cluster;         // CTAs per token (1 = none)
    int cpt;             // 16-byte chunks per thread per row (one-CTA kernels)
    int block;           // threads per CTA
    int grid_x;          // CTAs launched
    int early_trigger;   // signal dependents at kernel entry
};

// Fills *out, or returns an MFR_ERR_* code with a reason in err.  The caller
// has validated T, H, k and the option ranges.
inline int choose_launch(const PolicyIn& in, PolicyOut* out, char* err, size_t errn, int ring_threads) {
    const int chunks = static_cast<int>(in.H / 8);
    int variant = in.force_variant;
    int csize = in.cluster_size;
    if (in.fp4 && in.H % 16 != 0) {
        snprintf(err, errn, "NVFP4 output needs H %% 16 == 0 (H=%lld)", (long long)in.H);
        return MFR_ERR_UNSUPPORTED_SHAPE;
    }
    if (in.expert_norm) {
        // mfr_expert_norm.cu: a cluster of CTAs per token (small calls) or one
        // CTA per token, both holding the rows in registers when k <= 8; or the
        // ring kernel, which keeps a token's rows available until its slot
        // scales are known: k <= 8 and at most 4 column tiles (H <= 8192); two
        // tiles sit in registers and at most two stages are held, so two ring
        // stages suffice.
        const bool ring_ok = in.k <= 8 && in.H <= 8192 && in.stages >= 2;
        const bool regs_ok = in.k <= 8;
        if (variant == MFR_VARIANT_CLUSTER && !regs_ok) {
            snprintf(err, errn, "the per-expert RMSNorm cluster form holds at most 8 slots (k=%d)", in.k);
            return MFR_ERR_UNSUPPORTED_SHAPE;
        }
        if (variant == MFR_VARIANT_STREAM && !ring_ok) {
            snprintf(err, errn, "the per-expert RMSNorm ring kernel needs k <= 8 and H <= 8192");
            return MFR_ERR_UNSUPPORTED_SHAPE;
        }
        if (variant == MFR_VARIANT_AUTO) {
            const int64_t elems = in.T * in.H;
            if (regs_ok && elems <= kClusterMaxElems) {
                if (csize == 0) csize = en_cluster(chunks, elems);
                variant = csize > 1 ? MFR_VARIANT_CLUSTER : MFR_VARIANT_ROWS;
            } else {
                variant = (ring_ok && !rows_beats_ring(elems, false, in.sms)) ? MFR_VARIANT_STREAM
                                                                                 : MFR_VARIANT_ROWS;
            }
        }
    }
    if (variant == MFR_VARIANT_AUTO) {
        const int64_t elems = in.T * in.H;
        if (elems <= kClusterMaxElems) {
            if (csize == 0) {
                csize = in.fused ? decode_cluster(chunks, elems) : finalize_split(chunks, elems);
                // NVFP4 from 2^16 to 2^17 elements: CTAs of 64 threads (each CTA
                // also builds a 256-entry scale table; with 32-thread CTAs T = 32
                // at H = 4096 ran 3.01 us against 2.77 with 64, measured)
                if (in.fp4 && elems > (int64_t(1) << 16) && elems <= (int64_t(1) << 17))
                    csize = split_for_threads(chunks, 64);
            }
            variant = csize > 1 ? MFR_VARIANT_CLUSTER : MFR_VARIANT_ROWS;
        } else if (rows_beats_ring(elems, in.fp4, in.sms) || in.stages < 2) {
            variant = MFR_VARIANT_ROWS;
        } else {
            variant = MFR_VARIANT_STREAM;
        }
    } else if (variant == MFR_VARIANT_CLUSTER) {
        if (csize == 0) csize = auto_cluster(chunks);
        if (csize < 2) csize = 2;
    }
    if (variant != MFR_VARIANT_CLUSTER) csize = 1;
    // NVFP4 blocks of 16 columns must not straddle two CTAs of a cluster
    while (in.fp4 && csize > 1 && (chunks / csize) % 2 != 0) csize /= 2;
    if (variant == MFR_VARIANT_CLUSTER && csize < 2) variant = MFR_VARIANT_ROWS;

    PolicyOut o{};
    o.variant = variant;
    // Signal dependents at kernel entry only while this grid is small: a
    // large grid would let the next kernel park CTAs on every SM for the
    // whole call (the ring kernel never signals early, see mfr_stream.cu).
    o.early_trigger = (variant != MFR_VARIANT_STREAM && in.T * in.H <= kEarlyTriggerMaxElems) ? 1 : 0;
    if (variant == MFR_VARIANT_STREAM) {
        if (in.stages < 2) {
            snprintf(err, errn, "k=%d leaves room for fewer than 2 ring stages", in.k);
            return MFR_ERR_UNSUPPORTED_SHAPE;
        }
        o.cluster = 1;
        o.cpt = 1;
        o.block = ring_threads;
        o.grid_x = stream_grid(in.T, in.sms);
    } else {
        if (chunks % csize != 0) {
            snprintf(err, errn, "cluster of %d CTAs needs H/8 divisible by it (H=%lld)", csize, (long long)in.H);
            return MFR_ERR_UNSUPPORTED_SHAPE;
        }
        const int cta_chunks = chunks / csize;
        o.cluster = csize;
        o.cpt = pick_cpt(cta_chunks);
        if (o.cpt == 0) {
            snprintf(err, errn, "H=%lld too wide", (long long)in.H);
            return MFR_ERR_UNSUPPORTED_SHAPE;
        }
        o.block = round_up((cta_chunks + o.cpt - 1) / o.cpt, 32);
        o.grid_x = static_cast<int>(in.T > 0 ? in.T * csize : csize);
    }
    *out = o;
    return MFR_OK;
}

}  // namespace mfr
