// Device helpers shared by the kernels of this library (sm_103a only).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe_finalize_rmsnorm.h"

namespace mfr {

// ---- programmatic dependent launch ----------------------------------------
// Wait until every kernel this one depends on (the previous kernel in the
// stream, when launched with programmatic stream serialization) has finished
// and its writes are visible.  A no-op for an ordinary launch.
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Let the next kernel in the stream start its own prologue.  It still waits
// for this whole grid before reading what this grid writes.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Ask L2 to fetch `bytes` (multiple of 16, 16-byte aligned address) ahead of
// use.  A prefetch has no effect on what later loads return, so it may run
// before pdl_wait(): loads after the wait still see the producer's writes.
__device__ __forceinline__ void prefetch_l2_bulk(const void* ptr, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(ptr), "r"(bytes) : "memory");
}

// ---- loads and stores --------------------------------------------------------
// 16 bytes of read-once data, cached in L2 only (.cg): the rows were written
// by the previous kernel and, for few tokens, prefetched into L2 by the
// prologue.  volatile keeps it after pdl_wait().
__device__ __forceinline__ uint4 ld_stream_u4(const void* ptr) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(ptr));
    return v;
}

// 16 bytes of data this kernel may also write (the residual, in place).
__device__ __forceinline__ float4 ld_once_f4(const float* ptr) {
    float4 v;
    asm volatile("ld.global.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(ptr));
    return v;
}

__device__ __forceinline__ void st_f4(float* ptr, float4 v) {
    asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};"
                 :: "l"(ptr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w) : "memory");
}

__device__ __forceinline__ void st_u2(void* ptr, uint2 v) {
    asm volatile("st.global.v2.u32 [%0], {%1, %2};" :: "l"(ptr), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ void st_u4(void* ptr, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};"
                 :: "l"(ptr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// ---- shared-memory barriers and cluster stores ---------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

// Arrive once and announce `bytes` of asynchronous writes for this phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_test_parity(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done) : "r"(bar), "r"(parity) : "memory");
    return done != 0;
}

// Waits at most `limit` SM cycles for the phase with this parity to
// complete; false if it did not.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, long long limit) {
    if (mbar_test_parity(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_test_parity(bar, parity))
        if (clock64() - t0 > limit) return false;
    return true;
}

// Every wait of the kernels: bounded at ~2 s at 2 GHz.
constexpr long long kWaitCycles = 4000000000LL;
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    return mbar_wait_bounded(bar, parity, kWaitCycles);
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
    return remote;
}

// One-way 4-byte store into a peer CTA's shared memory; its arrival is
// counted (4 bytes) on the peer's mbarrier.
__device__ __forceinline__ void st_async_cluster_f32(uint32_t remote, float v, uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];"
                 :: "r"(remote), "r"(__float_as_uint(v)), "r"(remote_bar) : "memory");
}

// ---- bf16 -----------------------------------------------------------------------
// Element e (0..7) of 8 packed bf16 values, widened exactly to fp32.
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

// Two fp32 values rounded to nearest-even bf16, packed low = a, high = b.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// ---- NVFP4 ------------------------------------------------------------------------
// E4M3 byte of v: nearest-even, magnitudes beyond 448 saturate to 448.
__device__ __forceinline__ uint32_t e4m3_rn_sat(float v) {
    uint16_t e;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(e) : "f"(v));
    return e & 0xFFu;
}

// Value of an E4M3 byte (exact through f16).
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(b)));
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

// Two E2M1 codes (nearest-even, saturating at 6): lo in bits 3..0, hi in 7..4.
// The instruction puts its first source in the upper nibble.
__device__ __forceinline__ uint32_t e2m1x2_rn_sat(float lo, float hi) {
    uint16_t q;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
        : "=h"(q) : "f"(hi), "f"(lo));
    return q & 0xFFu;
}

// Byte index of the block scale of row t, block b (S blocks per row) in the
// NVFP4 output: row-major [T, S], or (tiled) the layout block-scaled FP4
// GEMMs read: the scale matrix padded to multiples of 128 rows and 4 columns
// is cut into 128 x 4 tiles of 512 consecutive bytes, tiles in row-major
// order, and scale (r, c) of a tile sits at byte (r mod 32) * 16 +
// ((r / 32) mod 4) * 4 + (c mod 4).
__device__ __forceinline__ int64_t nvfp4_sf_index(int64_t t, int b, int S, int tiled) {
    if (!tiled) return t * S + b;
    const int64_t tile = (t >> 7) * ((S + 3) >> 2) + (b >> 2);
    return tile * 512 + (t & 31) * 16 + ((t >> 5) & 3) * 4 + (b & 3);
}

// NVFP4 of a 16-element block held by a lane pair (lanes 2m and 2m+1, eight
// values each, lane 2m holding the first eight).  All 32 lanes must call it.
//   amax = max |y|;  sf = E4M3((amax / 6) * s_enc);  dec = value(sf) / s_enc;
//   enc = sf == 0 ? 0 : 1 / dec;  q_i = E2M1(y_i * enc)
// Every step is one correctly rounded FP32 operation; enc depends on sf
// alone, so it is read from enc_tab[sf], the 256 values computed once per
// call with the same two divisions.  Returns this lane's eight codes packed
// into 4 bytes (element 0 in the lowest nibble) and the scale byte in *sf.
__device__ __forceinline__ uint32_t nvfp4_block8(const float (&y)[8], float s_enc, const float* enc_tab,
                                                 uint32_t* sf) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(y[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    const uint32_t s8 = e4m3_rn_sat(__fmul_rn(__fdiv_rn(amax, 6.0f), s_enc));
    const float enc = enc_tab[s8];
    uint32_t w = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        w |= e2m1x2_rn_sat(__fmul_rn(y[2 * j], enc), __fmul_rn(y[2 * j + 1], enc)) << (8 * j);
    *sf = s8;
    return w;
}

// The same for a 16-element block held by a lane quad (lanes 4m..4m+3, four
// values each, in column order), with enc read from enc_tab[s8] (the 256
// values 1 / (value(s8) / s_enc) computed once per call, 0 at s8 = 0).
// Returns this lane's four codes in 2 bytes.
__device__ __forceinline__ uint32_t nvfp4_block4(const float (&y)[4], float s_enc, const float* enc_tab,
                                                 uint32_t* sf) {
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fabsf(y[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    const uint32_t s8 = e4m3_rn_sat(__fmul_rn(__fdiv_rn(amax, 6.0f), s_enc));
    const float enc = enc_tab[s8];
    const uint32_t w = e2m1x2_rn_sat(__fmul_rn(y[0], enc), __fmul_rn(y[1], enc)) |
                       (e2m1x2_rn_sat(__fmul_rn(y[2], enc), __fmul_rn(y[3], enc)) << 8);
    *sf = s8;
    return w;
}

// acc + b*b for a bf16 value b (its 16-bit pattern), one correctly rounded
// FP32 fused multiply-add taking b straight from the bf16 bits.  bf16 -> fp32
// is exact, so this equals fmaf(float(b), float(b), acc) (outputs checked
// bitwise equal on GB300); it saves the unpack instruction per element.
__device__ __forceinline__ float fma_bf16_sq(uint16_t b, float acc) {
    asm("fma.rn.f32.bf16 %0, %1, %1, %0;" : "+f"(acc) : "h"(b));
    return acc;
}

// Sum of squares of the four bf16 values in v (element 0 first) added to acc.
__device__ __forceinline__ float sumsq_bf16x4(uint2 v, float acc) {
    acc = fma_bf16_sq(static_cast<uint16_t>(v.x & 0xFFFFu), acc);
    acc = fma_bf16_sq(static_cast<uint16_t>(v.x >> 16), acc);
    acc = fma_bf16_sq(static_cast<uint16_t>(v.y & 0xFFFFu), acc);
    acc = fma_bf16_sq(static_cast<uint16_t>(v.y >> 16), acc);
    return acc;
}

// ---- reductions ------------------------------------------------------------------
// Butterfly sum over the 32 lanes.  Each level adds a value to its partner's,
// and fp32 addition is commutative, so every lane ends with the same bits.
__device__ __forceinline__ float warp_allreduce_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
    return v;
}

// Per-slot sums of 8 values over a warp in 9 shuffles: a reduce-scatter
// butterfly (xor 16, 8, 4 halve the slots a lane carries; xor 2, 1 finish)
// that returns the warp's sum of slot (lane >> 2) & 7 in lanes 4m..4m+3.
// The order of the additions is fixed, so the result is reproducible.
__device__ __forceinline__ float warp_reduce_scatter8(const float (&ss)[8], int lane) {
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
    float a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = b4 ? ss[i] : ss[i + 4];
        const float keep = b4 ? ss[i + 4] : ss[i];
        a[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 16);
    }
    float b[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = b3 ? a[i] : a[i + 2];
        const float keep = b3 ? a[i + 2] : a[i];
        b[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, 8);
    }
    float c = (b2 ? b[1] : b[0]) + __shfl_xor_sync(0xFFFFFFFFu, b2 ? b[0] : b[1], 4);
    c += __shfl_xor_sync(0xFFFFFFFFu, c, 2);
    c += __shfl_xor_sync(0xFFFFFFFFu, c, 1);
    return c;
}

}  // namespace mfr
