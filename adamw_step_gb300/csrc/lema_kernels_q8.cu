// lema_kernels_q8.cu -- the optimizer step and gradient accumulation with 8-bit
// moments and accumulators, sm_103a.
//
// Page "LEMA: Layer-wise Efficient Memory Abstraction", section "Quantization": the
// Adam moments and the gradient accumulators may be held as 8-bit integers and
// expanded to full precision only within each layer's AdamW update.  The
// arithmetic between decode and encode is the fp32 step of lema_kernels.cu, in the
// same order, with the same round-to-nearest intrinsics (built with --fmad=false,
// -ftz=false).
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "lema_device.cuh"
#include "lema_internal.h"
#include "lema_q8.h"

namespace lema {
namespace {

// ------------------------------------------------------------ 8-bit states
//
// Per 256-element block: one fp32 scale.  Signed fields (m, accumulator): scale =
// absmax / 127, code = rint(x * (127 / absmax)) clamped to [-127, 127].  The second
// moment as its root r = sqrt(v): scale = rmax / 255, code = min(ceil(r * (255 /
// rmax)), 255).  A block whose maximum is below 2^-100 is stored as zero.  Decoding
// multiplies code by scale.  Block maxima are exact, so the warp's shuffle reduction
// equals a sequential maximum.

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ void ld8_f32(const float* p, int valid, float (&x)[8]) {
    if (valid == 8) {
        const float4 a = ld_cs4(p), b = ld_cs4(p + 4);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = k < valid ? p[k] : 0.f;
    }
}

__device__ __forceinline__ void st8_f32(float* p, int valid, const float (&x)[8]) {
    if (valid == 8) {
        st_cs4(p, make_float4(x[0], x[1], x[2], x[3]));
        st_cs4(p + 4, make_float4(x[4], x[5], x[6], x[7]));
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (k < valid) p[k] = x[k];
    }
}

__device__ __forceinline__ void unpack8_bf16(const uint4& u, float (&x)[8]) {
    x[0] = bf16_lo(u.x); x[1] = bf16_hi(u.x); x[2] = bf16_lo(u.y); x[3] = bf16_hi(u.y);
    x[4] = bf16_lo(u.z); x[5] = bf16_hi(u.z); x[6] = bf16_lo(u.w); x[7] = bf16_hi(u.w);
}

__device__ __forceinline__ void ld8_bf16(const uint16_t* p, int valid, float (&x)[8]) {
    if (valid == 8) {
        unpack8_bf16(ld_cs8(p), x);
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = k < valid ? bf16_one(p + k) : 0.f;
    }
}

// Byte codes <-> floats without integer conversions.  Decoding places a code byte
// into the low mantissa bits of 2^23 (one byte permute) and subtracts 2^23, both
// exact; signed codes are first flipped to excess-128.  Encoding adds 1.5 * 2^23 to
// the fp32 value v: for |v| < 2^22 the sum lies in [2^23, 2^24), where the spacing is
// 1, so the single rounding of that add is round-half-even of v to an integer
// (= rint(v)), and the integer's two's-complement low byte is the code.
constexpr float kTwo23 = 8388608.0f;
constexpr float kRoundMagic = 12582912.0f;   // 1.5 * 2^23

// (2^23 + byte k of word) - offset, exact for offset 2^23 or 2^23 + 128.
__device__ __forceinline__ float byte_as_float(uint32_t word, int k, float offset) {
    // result bytes: [word byte k, 0x00, 0x00, 0x4B] = 2^23 + that byte
    return __uint_as_float(__byte_perm(word, 0x4B000000u, 0x7540u + uint32_t(k))) - offset;
}

// 8 one-byte codes as floats, exactly.  kSigned: int8 codes, else uint8.
// 8 one-byte codes held in two words, as floats, exactly.  kSigned: int8 codes.
template <bool kSigned>
__device__ __forceinline__ void decode8_codes(uint2 u, float (&q)[8]) {
    if (kSigned) {
        u.x ^= 0x80808080u;
        u.y ^= 0x80808080u;
    }
    const float offset = kSigned ? kTwo23 + 128.0f : kTwo23;   // excess-128 for int8
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        q[k] = byte_as_float(u.x, k, offset);
        q[k + 4] = byte_as_float(u.y, k, offset);
    }
}

template <bool kSigned, typename Byte>
__device__ __forceinline__ void ld8_codes(const Byte* p, int valid, float (&q)[8]) {
    uint2 u = make_uint2(0u, 0u);
    if (valid == 8) {
        u = __ldcs(reinterpret_cast<const uint2*>(p));
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t b = k < valid ? uint32_t(uint8_t(p[k])) : 0u;
            if (k < 4) u.x |= b << (8 * k);
            else u.y |= b << (8 * (k - 4));
        }
    }
    decode8_codes<kSigned>(u, q);
}

// Pack the low bytes of 8 integer-valued magic sums (see above) and store them.
template <typename Byte>
__device__ __forceinline__ void st8_codes(Byte* p, int valid, const float (&y)[8]) {
    uint32_t b[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) b[k] = __float_as_uint(y[k]);
    const uint32_t lo = __byte_perm(__byte_perm(b[0], b[1], 0x0040u), __byte_perm(b[2], b[3], 0x0040u), 0x5410u);
    const uint32_t hi = __byte_perm(__byte_perm(b[4], b[5], 0x0040u), __byte_perm(b[6], b[7], 0x0040u), 0x5410u);
    if (valid == 8) {
        __stcs(reinterpret_cast<uint2*>(p), make_uint2(lo, hi));
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (k < valid) p[k] = Byte((k < 4 ? lo >> (8 * k) : hi >> (8 * (k - 4))) & 0xFFu);
    }
}

// The scale of a block of signed values from its (exact) absolute maximum, and the
// factor 127/absmax that encodes it; tiny blocks are stored as zero.
__device__ __forceinline__ float signed_scale(float amax, float* inv) {
    if (amax < 0x1p-100f) amax = 0.f;
    const float s = __fdiv_rn(amax, 127.0f);
    *inv = s == 0.f ? 0.f : __fdiv_rn(127.0f, amax);
    return s;
}

// Encode the warp's block of signed values into magic sums y (code = low byte);
// returns the block scale.  |x| <= absmax and 127/absmax carries one rounding, so
// |x * (127/absmax)| < 127.0001 and rounds to at most 127: no clamp is needed.
__device__ __forceinline__ float encode_signed(const float (&x)[8], int valid, float (&y)[8]) {
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k)
        if (k < valid) amax = fmaxf(amax, fabsf(x[k]));
    float inv;
    const float s = signed_scale(warp_max(amax), &inv);
#pragma unroll
    for (int k = 0; k < 8; ++k) y[k] = __fadd_rn(__fmul_rn(x[k], inv), kRoundMagic);
    return s;
}

// The two block scales of the step (m: absmax / 127, sqrt(v): rmax / 255) and their
// encoding factors (127 / absmax, 255 / rmax; 0 for a zero block) from the warp's
// block maxima.  The four IEEE divides are independent, so lanes 0..3 each take one
// in a single pass of the divide and the warp reads them back by shuffle: the
// quotients are those of four separate divides.
__device__ __forceinline__ void step_scales(float amax, float rmax, int lane, float* m_scale,
                                            float* m_inv, float* r_scale, float* r_inv) {
    if (amax < 0x1p-100f) amax = 0.f;   // tiny blocks are stored as zero
    if (rmax < 0x1p-100f) rmax = 0.f;
    const int q = lane & 3;
    const float num = q == 0 ? amax : q == 1 ? 127.0f : q == 2 ? rmax : 255.0f;
    const float den = q == 0 ? 127.0f : q == 1 ? amax : q == 2 ? 255.0f : rmax;
    const float quo = __fdiv_rn(num, den);   // 127 / 0 = inf for a zero block: not used
    *m_scale = __shfl_sync(0xffffffffu, quo, 0);
    *r_scale = __shfl_sync(0xffffffffu, quo, 2);
    const float mi = __shfl_sync(0xffffffffu, quo, 1);
    const float ri = __shfl_sync(0xffffffffu, quo, 3);
    *m_inv = *m_scale == 0.f ? 0.f : mi;
    *r_inv = *r_scale == 0.f ? 0.f : ri;
}

// x / c rounded to nearest even, for the per-call constant c = sqrt(1 - beta2^t)
// given rc = RN(1/c), by Markstein's method (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Develop. 34(1),
// 1990): q0 = RN(x * rc) lies within one ulp of x/c, so the remainder x - c*q0 is
// an fp32 number that one fused multiply-add yields exactly, and RN(q0 + rem * rc)
// is then RN(x/c) -- the same result as an IEEE division, in three operations
// instead of a full divide.  It holds while nothing underflows or overflows: for
// x = 0, for 2^-100 <= x <= 2^64 (x/c and the remainder stay normal, since
// 2^-27 < c <= 1) and, fixed up below, for x = inf.  Here x = sqrt(v), which is
// never subnormal (the square root of the smallest positive fp32 number is 2^-74.5)
// and never above 2^64 (the square root of the largest).  NaN stays NaN.
__device__ __forceinline__ float div_by_const(float x, float c, float rc) {
    const float q0 = __fmul_rn(x, rc);
    const float rem = __fmaf_rn(-c, q0, x);
    const float q = __fmaf_rn(rem, rc, q0);
    return (x == 0.f || fabsf(x) == __int_as_float(0x7f800000)) ? q0 : q;   // +-0, +-inf
}

// The fp32 update on decoded states, as adamw_elem, also returning sqrt(v).
template <bool kPow2>
__device__ __forceinline__ void adamw_elem_q8(const StepScalars& s, float sum, float orig,
                                              float& w, float m_old, float r_old, float& m,
                                              float& root_v, float& delta) {
    const float g = kPow2 ? __fmul_rn(sum, s.inv_accum) : __fdiv_rn(sum, s.accum);
    float wn = __fmul_rn(w, s.decay);
    m = __fadd_rn(__fmul_rn(s.beta1, m_old), __fmul_rn(s.omb1, g));
    const float v_old = __fmul_rn(r_old, r_old);
    const float v = __fadd_rn(__fmul_rn(s.beta2, v_old), __fmul_rn(s.omb2, __fmul_rn(g, g)));
    root_v = __fsqrt_rn(v);
    const float den = __fadd_rn(div_by_const(root_v, s.bc2_sqrt, s.bc2_rcp), s.eps);
    wn = __fsub_rn(wn, __fmul_rn(s.step_size, __fdiv_rn(m, den)));
    w = wn;
    delta = __fsub_rn(wn, orig);
}

// A lane's 8 elements of its warp's 256-element block are either 8 consecutive ones
// at e (kSplit = false: any `valid`) or two runs of 4, at e and e + 128 (kSplit =
// true, whole groups only: lane l takes 4l..4l+3 and 128+4l..128+4l+3, so that a
// warp's shared-memory reads are conflict-free and each store instruction writes
// one contiguous span).  Elementwise results do not depend on the split, and the
// block maxima are over the same 256 elements.
template <bool kSplit>
__device__ __forceinline__ void put8_f32(float* p, int valid, const float (&x)[8]) {
    if (kSplit) {
        st_cs4(p, make_float4(x[0], x[1], x[2], x[3]));
        st_cs4(p + 128, make_float4(x[4], x[5], x[6], x[7]));
    } else {
        st8_f32(p, valid, x);
    }
}

template <bool kSplit>
__device__ __forceinline__ void put8_bf16(uint16_t* p, int valid, const float (&x)[8]) {
    if (kSplit || valid == 8) {
        uint4 b;
        b.x = bf16x2_rne(x[0], x[1]);
        b.y = bf16x2_rne(x[2], x[3]);
        b.z = bf16x2_rne(x[4], x[5]);
        b.w = bf16x2_rne(x[6], x[7]);
        if (kSplit) {
            __stcs(reinterpret_cast<uint2*>(p), make_uint2(b.x, b.y));
            __stcs(reinterpret_cast<uint2*>(p + 128), make_uint2(b.z, b.w));
        } else {
            st_cs8(p, b);
        }
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (k < valid) p[k] = bf16_rne(x[k]);
    }
}

template <bool kSplit, typename Byte>
__device__ __forceinline__ void put8_codes(Byte* p, int valid, const float (&y)[8]) {
    if (kSplit) {
        uint32_t b[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) b[k] = __float_as_uint(y[k]);
        const uint32_t lo = __byte_perm(__byte_perm(b[0], b[1], 0x0040u), __byte_perm(b[2], b[3], 0x0040u), 0x5410u);
        const uint32_t hi = __byte_perm(__byte_perm(b[4], b[5], 0x0040u), __byte_perm(b[6], b[7], 0x0040u), 0x5410u);
        __stcs(reinterpret_cast<unsigned int*>(p), lo);
        __stcs(reinterpret_cast<unsigned int*>(p + 128), hi);
    } else {
        st8_codes(p, valid, y);
    }
}

// Outputs of one lane's 8 elements of a 256-element block from their decoded inputs:
// the update in the documented order, master/delta/w stored, m and sqrt(v)
// re-encoded with the warp's block scales, the accumulator reset when asked.  w[]
// enters as master and leaves as the new master.
template <bool kPow2, bool kSplit>
__device__ __forceinline__ void step_group_q8(const StepScalars& s, const StepDescQ8* dp, int64_t e,
                                              int64_t blk, int lane, int valid, bool zero_acc,
                                              float (&w)[8], const float (&mq)[8], float ms,
                                              const float (&rq)[8], float rs,
                                              const float (&sum)[8], const float (&orig)[8]) {
    float m[8], root_v[8], d[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
        adamw_elem_q8<kPow2>(s, sum[k], orig[k], w[k], __fmul_rn(mq[k], ms), __fmul_rn(rq[k], rs),
                             m[k], root_v[k], d[k]);

    put8_f32<kSplit>(dp->master_out + e, valid, w);
    put8_f32<kSplit>(dp->delta + e, valid, d);
    put8_bf16<kSplit>(dp->w + e, valid, w);
    float amax = 0.f, rmax = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k)
        if (k < valid) {
            amax = fmaxf(amax, fabsf(m[k]));
            rmax = fmaxf(rmax, root_v[k]);
        }
    float m_scale, m_inv, r_scale, r_inv;
    step_scales(warp_max(amax), warp_max(rmax), lane, &m_scale, &m_inv, &r_scale, &r_inv);
    // m: rint(m * 127/absmax) (|code| <= 127 without a clamp, as in encode_signed);
    // sqrt(v): its root rounded up and capped at 255
    float y[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) y[k] = __fadd_rn(__fmul_rn(m[k], m_inv), kRoundMagic);
    put8_codes<kSplit>(dp->m_q_out + e, valid, y);
#pragma unroll
    for (int k = 0; k < 8; ++k)
        y[k] = __fadd_rn(fminf(ceilf(__fmul_rn(root_v[k], r_inv)), 255.f), kRoundMagic);
    put8_codes<kSplit>(dp->r_q_out + e, valid, y);
    if (lane == 0) {
        dp->m_scale_out[blk] = m_scale;
        dp->r_scale_out[blk] = r_scale;
    }
    if (zero_acc) {
        const float z[8] = {kRoundMagic, kRoundMagic, kRoundMagic, kRoundMagic,
                            kRoundMagic, kRoundMagic, kRoundMagic, kRoundMagic};
        put8_codes<kSplit>(dp->acc_q + e, valid, z);
        if (lane == 0) dp->acc_scale[blk] = 0.f;
    }
}

// ---- persistent kernels: groups of 2048 elements streamed through shared memory
//
// The step's arithmetic needs ~80 registers a thread, which leaves too few warps to
// hide HBM latency with plain loads.  So the loads are decoupled from the warps: each
// CTA (4 per SM, 64 registers a thread) walks its share of the launch's groups (2048 elements = one lane-group of 8 for each of the 256 threads) and keeps
// the next groups' inputs in flight as bulk asynchronous copies into a ring of
// shared-memory buffers, one mbarrier each.  A group that is not wholly inside its
// tensor (the ragged end) is read with plain loads instead; its barrier phase is
// completed by a plain arrival so that the ring's phase bookkeeping stays uniform.
constexpr int kGroup = kThreads * kVec;                       // elements per group
constexpr int kGroupsPerChunk = kIters;
constexpr int kOffMaster = 0;                                 // fp32
constexpr int kOffMq = kOffMaster + 4 * kGroup;               // int8
constexpr int kOffRq = kOffMq + kGroup;                       // uint8
constexpr int kOffAq = kOffRq + kGroup;                       // int8
constexpr int kOffGrad = kOffAq + kGroup;                     // bf16
constexpr int kOffOrig = kOffGrad + 2 * kGroup;               // bf16
constexpr int kScaleBytes = 4 * kGroup / kQBlock;             // one group's scales of a field
constexpr int kOffMs = kOffOrig + 2 * kGroup;                 // fp32 scales of m, sqrt(v), acc
constexpr int kOffRs = kOffMs + kScaleBytes;
constexpr int kOffAs = kOffRs + kScaleBytes;
constexpr int kStepStageBytes = kOffMs + 128;                 // 22656 (128-byte multiple)
constexpr int kStepBufs = 2;
constexpr int kStepSmem = kStepBufs * kStepStageBytes;        // 45312
static_assert(kScaleBytes == 32 && kOffAs + kScaleBytes <= kStepStageBytes, "scale slots");
constexpr int kStepCtasPerSm = 4;   // 4 x (256 threads, 45 KB ring) per SM
static_assert(kStepStageBytes % 128 == 0, "buffers stay 128-byte aligned");
static_assert(kGroup == 8 * kQBlock, "a group is whole quantization blocks");

// Kernel-side bounded waits that ran out (read by lema_kernel_wait_timeouts).
__device__ unsigned long long g_wait_timeouts = 0;

// How long a wait for a group's staged inputs may take before the CTA gives up.
// The copies of one 22 KB group take microseconds, so the default of 1 s is only
// reached when something is wrong.  A test hook may lower it (0: give up at the
// first poll that finds the copies still in flight) to exercise the give-up path.
constexpr uint64_t kWaitNs = 1000000000ull;
__device__ unsigned long long g_wait_limit_ns = kWaitNs;
// After a give-up, the CTA still waits for the copies it has issued before its
// shared memory goes away; that drain has its own, longer bound, which the test
// hook does not change.
constexpr uint64_t kDrainNs = 10000000000ull;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of parity `parity` of an mbarrier to complete, giving up after
// about `limit_ns` (limit_ns == 0: one non-blocking test, no wait).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (limit_ns == 0) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}"
            : "=r"(done) : "r"(bar), "r"(parity) : "memory");
        return done != 0;
    }
    uint64_t start = 0;
    for (uint32_t i = 0;; ++i) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}"
            : "=r"(done) : "r"(bar), "r"(parity) : "memory");
        if (done) return true;
        if ((i & 63) == 0) {
            const uint64_t now = global_ns();
            if (i == 0) start = now;
            else if (now - start > limit_ns) return false;
        }
    }
}

struct Group {
    const StepDescQ8* dp;
    int64_t begin;   // first element of the group in its tensor
    bool full;       // all kGroup elements inside the tensor
    bool empty;      // none inside
};

__device__ __forceinline__ Group group_of(const StepDescQ8* descs, const Chunk* chunks, int64_t w) {
    const Chunk c = chunks[w / kGroupsPerChunk];
    Group g;
    g.dp = descs + c.tensor;
    g.begin = c.begin + (w % kGroupsPerChunk) * kGroup;
    const int64_t n = g.dp->n;
    g.full = g.begin + kGroup <= n;
    g.empty = g.begin >= n;
    return g;
}

// Thread 0: start group w's copies into buffer `buf` (or, for a group that is not
// whole, complete the barrier's phase without data).
__device__ __forceinline__ void issue_group(const Group& g, unsigned char* buf, uint32_t bar) {
    if (!g.full) {
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
        return;
    }
    const StepDescQ8* dp = g.dp;
    const bool has_acc = dp->acc_q != nullptr, has_grad = dp->grad != nullptr;
    const uint32_t tx = kGroup * (4 + 1 + 1 + 2) + 2 * kScaleBytes +
                        (has_acc ? kGroup + kScaleBytes : 0) + (has_grad ? 2 * kGroup : 0);
    const uint32_t st = smem_addr(buf);
    const int64_t g0 = g.begin;
    const int64_t b0 = g0 / kQBlock;   // a multiple of 8: the scale slices start 32-byte aligned
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(tx)
                 : "memory");
    bulk_load(st + kOffMaster, dp->master_in + g0, 4 * kGroup, bar);
    bulk_load(st + kOffMq, dp->m_q_in + g0, kGroup, bar);
    bulk_load(st + kOffRq, dp->r_q_in + g0, kGroup, bar);
    if (has_acc) bulk_load(st + kOffAq, dp->acc_q + g0, kGroup, bar);
    if (has_grad) bulk_load(st + kOffGrad, dp->grad + g0, 2 * kGroup, bar);
    bulk_load(st + kOffOrig, dp->orig + g0, 2 * kGroup, bar);
    bulk_load(st + kOffMs, dp->m_scale_in + b0, kScaleBytes, bar);
    bulk_load(st + kOffRs, dp->r_scale_in + b0, kScaleBytes, bar);
    if (has_acc) bulk_load(st + kOffAs, dp->acc_scale + b0, kScaleBytes, bar);
}

// One whole group from shared memory, lanes split as in step_group_q8<.., true>.
template <bool kPow2>
__device__ __forceinline__ void step_staged(const StepScalars& s, const Group& g,
                                            const unsigned char* st, int lane) {
    const StepDescQ8* dp = g.dp;
    const int wb = (threadIdx.x >> 5) * kQBlock;       // the warp's block within the group
    const int a = wb + 4 * lane, b = a + 128;           // the lane's two runs of 4
    const int64_t e = g.begin + a;
    const int64_t blk = (g.begin + wb) / kQBlock;
    const bool has_acc = dp->acc_q != nullptr;
    const int wq = 4 * (threadIdx.x >> 5);               // the warp's scale, in bytes
    const float ms = *reinterpret_cast<const float*>(st + kOffMs + wq);
    const float rs = *reinterpret_cast<const float*>(st + kOffRs + wq);
    const float as = has_acc ? *reinterpret_cast<const float*>(st + kOffAs + wq) : 0.f;
    auto codes = [&](int off) {
        return make_uint2(*reinterpret_cast<const uint32_t*>(st + off + a),
                          *reinterpret_cast<const uint32_t*>(st + off + b));
    };
    auto bf16s = [&](int off) {
        const uint2 x = *reinterpret_cast<const uint2*>(st + off + 2 * a);
        const uint2 y = *reinterpret_cast<const uint2*>(st + off + 2 * b);
        return make_uint4(x.x, x.y, y.x, y.y);
    };
    float w[8], mq[8], rq[8], sum[8], orig[8];
    const float4 w0 = *reinterpret_cast<const float4*>(st + kOffMaster + 4 * a);
    const float4 w1 = *reinterpret_cast<const float4*>(st + kOffMaster + 4 * b);
    w[0] = w0.x; w[1] = w0.y; w[2] = w0.z; w[3] = w0.w;
    w[4] = w1.x; w[5] = w1.y; w[6] = w1.z; w[7] = w1.w;
    decode8_codes<true>(codes(kOffMq), mq);
    decode8_codes<false>(codes(kOffRq), rq);
    if (has_acc) {
        decode8_codes<true>(codes(kOffAq), sum);
#pragma unroll
        for (int k = 0; k < 8; ++k) sum[k] = __fmul_rn(sum[k], as);
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) sum[k] = 0.f;
    }
    if (dp->grad) {
        float gr[8];
        unpack8_bf16(bf16s(kOffGrad), gr);
#pragma unroll
        for (int k = 0; k < 8; ++k) sum[k] = __fadd_rn(sum[k], gr[k]);
    }
    unpack8_bf16(bf16s(kOffOrig), orig);
    step_group_q8<kPow2, true>(s, dp, e, blk, lane, 8, (dp->flags & kZeroAcc) != 0, w, mq, ms, rq,
                               rs, sum, orig);
}

// One group with plain loads (the ragged end of a tensor).
template <bool kPow2>
__device__ __forceinline__ void step_direct(const StepScalars& s, const Group& g, int lane) {
    const StepDescQ8* dp = g.dp;
    const int64_t end = dp->n;
    const int64_t e = g.begin + int64_t(threadIdx.x) * kVec;
    const int64_t block_start = e - int64_t(lane) * kVec;
    if (block_start >= end) return;   // the whole warp is past the tensor's end
    const int64_t blk = block_start / kQBlock;
    const int valid = int(max(int64_t(0), min(int64_t(kVec), end - e)));
    float w[8], sum[8], orig[8], gr[8];
    float mq[8], rq[8], aq[8];
    ld8_f32(dp->master_in + e, valid, w);
    ld8_codes<true>(dp->m_q_in + e, valid, mq);
    ld8_codes<false>(dp->r_q_in + e, valid, rq);
    const float ms = dp->m_scale_in[blk];
    const float rs = dp->r_scale_in[blk];
    if (dp->acc_q) {
        ld8_codes<true>(dp->acc_q + e, valid, aq);
        const float as = dp->acc_scale[blk];
#pragma unroll
        for (int k = 0; k < 8; ++k) sum[k] = __fmul_rn(aq[k], as);
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) sum[k] = 0.f;
    }
    if (dp->grad) {
        ld8_bf16(dp->grad + e, valid, gr);
#pragma unroll
        for (int k = 0; k < 8; ++k) sum[k] = __fadd_rn(sum[k], gr[k]);
    }
    ld8_bf16(dp->orig + e, valid, orig);
    step_group_q8<kPow2, false>(s, dp, e, blk, lane, valid, (dp->flags & kZeroAcc) != 0, w, mq,
                                ms, rq, rs, sum, orig);
}

// The persistent ring loop (the 8-bit step's; written for any Op).  CTA b takes
// groups b, b + G, b + 2G, ... (G = gridDim.x) of the launch's n_groups; Op gives the
// group of an index, starts a group's copies into a buffer (thread 0), and runs a
// group from a buffer (whole groups) or with plain loads (the rest).  Buffer j has
// one mbarrier; after a group every thread meets at a CTA barrier and thread 0
// refills the buffer with the group Op::kBufs steps ahead.
//
// A wait that runs out stops the CTA: it counts the event in g_wait_timeouts, sets
// *gave_up (a word in host-mapped memory the host library reads after the launch has
// finished; may be null), waits (bounded by kDrainNs) for the copies it has issued,
// and returns.  The groups it had not finished keep their old outputs.
template <typename Op>
__device__ __forceinline__ void ring_run(const Op& op, int64_t n_groups, unsigned int* gave_up) {
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t bars[Op::kBufs];
    const int lane = threadIdx.x & 31;
    const int64_t G = gridDim.x;

    if (threadIdx.x == 0) {
        for (int j = 0; j < Op::kBufs; ++j)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&bars[j]))
                         : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        for (int j = 0; j < Op::kBufs; ++j) {
            const int64_t w = blockIdx.x + j * G;
            if (w < n_groups)
                op.issue(op.group(w), ring + j * Op::kStageBytes, smem_addr(&bars[j]));
        }
    }
    __syncthreads();   // barriers initialized before anyone waits on them

    const uint64_t limit_ns = *const_cast<const volatile unsigned long long*>(&g_wait_limit_ns);
    int64_t k = 0;
    for (int64_t w = blockIdx.x; w < n_groups; w += G, ++k) {
        const int j = int(k % Op::kBufs);
        const uint32_t parity = uint32_t((k / Op::kBufs) & 1);
        const auto g = op.group(w);
        const bool ok = wait_phase(smem_addr(&bars[j]), parity, limit_ns);
        if (ok && !g.empty) {
            if (g.full) op.staged(g, ring + j * Op::kStageBytes, lane);
            else op.direct(g, lane);
        }
        // every thread is done with buffer j (or some wait ran out) ...
        if (__syncthreads_or(!ok)) {
            // Record it, let the copies still in flight land (again bounded) before
            // the CTA's shared memory goes away, and stop.
            if (threadIdx.x == 0) {
                atomicAdd(&g_wait_timeouts, 1ull);
                if (gave_up) {
                    *reinterpret_cast<volatile unsigned int*>(gave_up) = 1u;
                    __threadfence_system();
                }
                // The groups issued and not yet consumed: k .. k + kBufs - 1.
                for (int64_t q = 0; q < Op::kBufs; ++q) {
                    const int64_t kq = k + q;
                    if (blockIdx.x + kq * G >= n_groups) break;
                    wait_phase(smem_addr(&bars[kq % Op::kBufs]), uint32_t((kq / Op::kBufs) & 1),
                               kDrainNs);
                }
            }
            return;
        }
        // ... so thread 0 refills it with the group kBufs steps ahead (after the
        // threads' reads, ordered before the asynchronous copies' writes).
        if (threadIdx.x == 0) {
            const int64_t wn = w + Op::kBufs * G;
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            if (wn < n_groups)
                op.issue(op.group(wn), ring + j * Op::kStageBytes, smem_addr(&bars[j]));
        }
    }
}

template <bool kPow2>
struct StepOp {
    static constexpr int kBufs = kStepBufs;
    static constexpr int kStageBytes = kStepStageBytes;
    const StepDescQ8* descs;
    const Chunk* chunks;
    StepScalars s;
    __device__ Group group(int64_t w) const { return group_of(descs, chunks, w); }
    __device__ void issue(const Group& g, unsigned char* buf, uint32_t bar) const {
        issue_group(g, buf, bar);
    }
    __device__ void staged(const Group& g, const unsigned char* buf, int lane) const {
        step_staged<kPow2>(s, g, buf, lane);
    }
    __device__ void direct(const Group& g, int lane) const { step_direct<kPow2>(s, g, lane); }
};

template <bool kPow2>
__global__ void __launch_bounds__(kThreads, kStepCtasPerSm)
adamw_q8_kernel(const StepDescQ8* __restrict__ descs, const Chunk* __restrict__ chunks,
                int64_t n_groups, const StepScalars s, unsigned int* gave_up) {
    ring_run(StepOp<kPow2>{descs, chunks, s}, n_groups, gave_up);
}

__device__ __forceinline__ void accum_q8_chunk(const AccDescQ8* __restrict__ dp, const Chunk c) {
    const int64_t end = min(c.begin + kChunk, dp->n);
    const int lane = threadIdx.x & 31;

    if (c.begin + kChunk <= dp->n) {
        // A whole chunk (32 blocks): warp w owns blocks 4w..4w+3, eight lanes to a
        // block; lane l takes elements 8(l mod 8) + 64j .. +7 (j = 0..3) of block
        // 4w + l/8.  The per-block work (maximum over the block, scale, reciprocal)
        // then runs once per warp for four blocks, and each load or store instruction
        // of the warp still covers four whole 64-element runs.  Every load is issued
        // before any is used.
        static_assert(kChunk == 32 * kQBlock && kIters * 64 == kQBlock, "chunk = 8 warps x 4 blocks");
        const int8_t* acc_in = dp->acc_q_in;
        const int64_t blk0 = c.begin + int64_t(4 * (threadIdx.x >> 5) + (lane >> 3)) * kQBlock;
        const int sub = (lane & 7) * kVec;
        uint4 graw[kIters];
        uint2 codes[kIters];
        float sc = 0.f;
#pragma unroll
        for (int j = 0; j < kIters; ++j) {
            const int64_t e = blk0 + 64 * j + sub;
            graw[j] = ld_cs8(dp->grad + e);
            if (acc_in) codes[j] = __ldcs(reinterpret_cast<const uint2*>(acc_in + e));
        }
        if (acc_in) sc = dp->acc_scale_in[blk0 / kQBlock];
        float a[kIters][8];
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < kIters; ++j) {
            float g[8];
            if (acc_in) {
                decode8_codes<true>(codes[j], a[j]);
#pragma unroll
                for (int k = 0; k < 8; ++k) a[j][k] = __fmul_rn(a[j][k], sc);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) a[j][k] = 0.f;
            }
            unpack8_bf16(graw[j], g);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                a[j][k] = __fadd_rn(a[j][k], g[k]);
                amax = fmaxf(amax, fabsf(a[j][k]));
            }
        }
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        float inv;
        const float scale = signed_scale(amax, &inv);
#pragma unroll
        for (int j = 0; j < kIters; ++j) {
            float y[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) y[k] = __fadd_rn(__fmul_rn(a[j][k], inv), kRoundMagic);
            st8_codes(dp->acc_q_out + blk0 + 64 * j + sub, 8, y);
        }
        if ((lane & 7) == 0) dp->acc_scale_out[blk0 / kQBlock] = scale;
        return;
    }

#pragma unroll 1
    for (int it = 0; it < kIters; ++it) {
        const int64_t e = c.begin + (int64_t(it) * kThreads + threadIdx.x) * kVec;
        const int64_t block_start = e - int64_t(lane) * kVec;
        if (block_start >= end) continue;
        const int64_t blk = block_start / kQBlock;
        const int valid = int(max(int64_t(0), min(int64_t(kVec), end - e)));
        float a[8], g[8];
        if (dp->acc_q_in) {
            float aq[8];
            ld8_codes<true>(dp->acc_q_in + e, valid, aq);
            const float as = dp->acc_scale_in[blk];
#pragma unroll
            for (int k = 0; k < 8; ++k) a[k] = __fmul_rn(aq[k], as);
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) a[k] = 0.f;
        }
        ld8_bf16(dp->grad + e, valid, g);
#pragma unroll
        for (int k = 0; k < 8; ++k) a[k] = __fadd_rn(a[k], g[k]);
        float y[8];
        const float scale = encode_signed(a, valid, y);
        st8_codes(dp->acc_q_out + e, valid, y);
        if (lane == 0) dp->acc_scale_out[blk] = scale;
    }
}

__global__ void __launch_bounds__(kThreads)
accum_q8_kernel(const AccDescQ8* __restrict__ descs, const Chunk* __restrict__ chunks) {
    const Chunk c = chunks[blockIdx.x];
    accum_q8_chunk(descs + c.tensor, c);
}

template <int N>
__global__ void __launch_bounds__(kThreads)
accum_q8_kernel_v(const __grid_constant__ DescTable<AccDescQ8, N> t, const Chunk* __restrict__ chunks) {
    const Chunk c = chunks[blockIdx.x];
    accum_q8_chunk(&t.d[c.tensor], c);
}

template <bool kPow2, int N>
__global__ void __launch_bounds__(kThreads, kStepCtasPerSm)
adamw_q8_kernel_v(const __grid_constant__ DescTable<StepDescQ8, N> t, const Chunk* __restrict__ chunks,
                  int64_t n_groups, const StepScalars s, unsigned int* gave_up) {
    ring_run(StepOp<kPow2>{&t.d[0], chunks, s}, n_groups, gave_up);
}

}  // namespace

namespace {

// Per device, once: the step's ring exceeds the 48 KB default of dynamic shared
// memory, and its persistent grid is sized by the SM count.
template <typename K>
cudaError_t opt_in(K kernel) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kStepSmem);
}

cudaError_t ring_setup(int* n_sm) {
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static int sms[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(mu);
    if (sms[dev] == 0) {
        const cudaError_t r[] = {
            opt_in(adamw_q8_kernel<true>), opt_in(adamw_q8_kernel<false>),
            opt_in(adamw_q8_kernel_v<true, kValueTableSmall>),
            opt_in(adamw_q8_kernel_v<false, kValueTableSmall>),
            opt_in(adamw_q8_kernel_v<true, kValueTableMax>),
            opt_in(adamw_q8_kernel_v<false, kValueTableMax>)};
        for (cudaError_t x : r)
            if (x != cudaSuccess) return x;
        int count = 0;
        e = cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        sms[dev] = count;
    }
    *n_sm = sms[dev];
    return cudaSuccess;
}

template <typename D, int N>
DescTable<D, N> table_of(const D* host, int32_t count) {
    DescTable<D, N> t;
    std::memset(&t, 0, sizeof t);
    std::memcpy(t.d, host, sizeof(D) * size_t(count));
    return t;
}

}  // namespace

cudaError_t launch_accum_q8(const AccDescQ8* descs, const Chunk* chunks, int64_t n_chunks,
                            cudaStream_t stream) {
    if (n_chunks <= 0) return cudaSuccess;
    accum_q8_kernel<<<dim3(unsigned(n_chunks)), kThreads, 0, stream>>>(descs, chunks);
    return cudaGetLastError();
}

cudaError_t launch_step_q8(const StepDescQ8* descs, const Chunk* chunks, int64_t n_chunks,
                           const StepScalars& s, unsigned int* gave_up, cudaStream_t stream) {
    if (n_chunks <= 0) return cudaSuccess;
    int n_sm = 0;
    const cudaError_t e = ring_setup(&n_sm);
    if (e != cudaSuccess) return e;
    const int64_t n_groups = n_chunks * kGroupsPerChunk;
    const unsigned grid = unsigned(std::min<int64_t>(n_groups, int64_t(n_sm) * kStepCtasPerSm));
    if (s.accum_pow2)
        adamw_q8_kernel<true><<<grid, kThreads, kStepSmem, stream>>>(descs, chunks, n_groups, s,
                                                                     gave_up);
    else
        adamw_q8_kernel<false><<<grid, kThreads, kStepSmem, stream>>>(descs, chunks, n_groups, s,
                                                                      gave_up);
    return cudaGetLastError();
}

cudaError_t launch_accum_q8_v(const AccDescQ8* host_descs, int32_t count, const Chunk* chunks,
                              int64_t n_chunks, cudaStream_t stream) {
    if (n_chunks <= 0) return cudaSuccess;
    if (count > kValueTableMax) return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>(n_chunks));
    if (count <= kValueTableSmall)
        accum_q8_kernel_v<kValueTableSmall><<<grid, kThreads, 0, stream>>>(
            table_of<AccDescQ8, kValueTableSmall>(host_descs, count), chunks);
    else
        accum_q8_kernel_v<kValueTableMax><<<grid, kThreads, 0, stream>>>(
            table_of<AccDescQ8, kValueTableMax>(host_descs, count), chunks);
    return cudaGetLastError();
}

cudaError_t launch_step_q8_v(const StepDescQ8* host_descs, int32_t count, const Chunk* chunks,
                             int64_t n_chunks, const StepScalars& s, unsigned int* gave_up,
                             cudaStream_t stream) {
    if (n_chunks <= 0) return cudaSuccess;
    if (count > kValueTableMax) return cudaErrorInvalidValue;
    int n_sm = 0;
    const cudaError_t e = ring_setup(&n_sm);
    if (e != cudaSuccess) return e;
    const int64_t n_groups = n_chunks * kGroupsPerChunk;
    const dim3 grid(static_cast<unsigned>(std::min<int64_t>(n_groups, int64_t(n_sm) * kStepCtasPerSm)));
    if (count <= kValueTableSmall) {
        const auto t = table_of<StepDescQ8, kValueTableSmall>(host_descs, count);
        if (s.accum_pow2)
            adamw_q8_kernel_v<true, kValueTableSmall><<<grid, kThreads, kStepSmem, stream>>>(t, chunks, n_groups, s, gave_up);
        else
            adamw_q8_kernel_v<false, kValueTableSmall><<<grid, kThreads, kStepSmem, stream>>>(t, chunks, n_groups, s, gave_up);
    } else {
        const auto t = table_of<StepDescQ8, kValueTableMax>(host_descs, count);
        if (s.accum_pow2)
            adamw_q8_kernel_v<true, kValueTableMax><<<grid, kThreads, kStepSmem, stream>>>(t, chunks, n_groups, s, gave_up);
        else
            adamw_q8_kernel_v<false, kValueTableMax><<<grid, kThreads, kStepSmem, stream>>>(t, chunks, n_groups, s, gave_up);
    }
    return cudaGetLastError();
}

namespace {

// Every x >= 0 from bit pattern `first` on (grid-stride), div_by_const against the
// IEEE division; counts mismatches inside the domain div_by_const is used on (x = 0,
// 2^-100 <= x <= 2^64, inf, NaN) and, separately, outside it (subnormal or tiny x,
// and finite x above 2^64, where x/c may overflow).
__global__ void check_div_by_const_kernel(float c, float rc, uint32_t first, uint32_t last,
                                          unsigned long long* bad) {
    unsigned long long in_dom = 0, out_dom = 0;
    for (uint64_t b = first + uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; b <= last;
         b += uint64_t(gridDim.x) * blockDim.x) {
        const float x = __uint_as_float(uint32_t(b));
        const float want = __fdiv_rn(x, c), got = div_by_const(x, c, rc);
        const bool same = __float_as_uint(want) == __float_as_uint(got) ||
                          (want != want && got != got);
        if (!same) {
            const bool tiny = x != 0.f && x < 0x1p-100f;
            const bool huge = x > 0x1p64f && x <= __int_as_float(0x7f7fffff);
            if (tiny || huge) ++out_dom;
            else ++in_dom;
        }
    }
    if (in_dom) atomicAdd(&bad[0], in_dom);
    if (out_dom) atomicAdd(&bad[1], out_dom);
}

}  // namespace

cudaError_t check_div_by_const(float c, float rc, unsigned long long* bad_dev,
                               cudaStream_t stream) {
    check_div_by_const_kernel<<<1216, 256, 0, stream>>>(c, rc, 0u, 0x7fffffffu, bad_dev);
    return cudaGetLastError();
}

cudaError_t read_wait_timeouts(unsigned long long* out) {
    return cudaMemcpyFromSymbol(out, g_wait_timeouts, sizeof(*out));
}

cudaError_t set_wait_limit(int64_t ns) {
    const unsigned long long v = ns < 0 ? kWaitNs : static_cast<unsigned long long>(ns);
    return cudaMemcpyToSymbol(g_wait_limit_ns, &v, sizeof v);
}

}  // namespace lema
