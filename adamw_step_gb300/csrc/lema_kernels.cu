// lema_kernels.cu -- the two HBM-bound kernels of the optimizer step with fp32
// states, the delta merge, and the table install, sm_103a (8-bit states:
// lema_kernels_q8.cu).
//
// Page "LEMA: Layer-wise Efficient Memory Abstraction", section "Selective Full
// Fine-Tuning": fp32 gradient accumulation, per-layer AdamW on fp32 states, fp32
// delta (updated - original); section "Quick Start": torch.optim.AdamW semantics.
//
// Nothing here is a contraction, so there is no tensor-core work: both kernels are
// bound by HBM bandwidth (accumulate 10 B/element, step 40 B/element).  Each CTA
// owns one chunk of one tensor (chunk map built on the host); every thread moves 8
// consecutive elements per iteration with 16-byte loads and stores marked
// evict-first (.cs), since every byte is touched exactly once per launch.
//
// Arithmetic: explicit round-to-nearest intrinsics (__fmul_rn, __fadd_rn,
// __fdiv_rn, __fsqrt_rn) so that nothing is contracted into an FMA and the
// operation order is exactly the one documented in lema.h; the file is also built
// with --fmad=false, -ftz=false, IEEE division and square root.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "lema_device.cuh"
#include "lema_internal.h"

namespace lema {
namespace {


// The element update, in the documented order.  K a power of two: acc * (1/K) is
// the same correctly rounded quotient as acc / K (the exact values coincide).
template <bool kPow2>
__device__ __forceinline__ void adamw_elem(const StepScalars& s, float acc, float orig,
                                           float& w, float& m, float& v, float& delta) {
    const float g = kPow2 ? __fmul_rn(acc, s.inv_accum) : __fdiv_rn(acc, s.accum);
    float wn = __fmul_rn(w, s.decay);
    const float mn = __fadd_rn(__fmul_rn(s.beta1, m), __fmul_rn(s.omb1, g));
    const float vn = __fadd_rn(__fmul_rn(s.beta2, v), __fmul_rn(s.omb2, __fmul_rn(g, g)));
    const float den = __fadd_rn(__fdiv_rn(__fsqrt_rn(vn), s.bc2_sqrt), s.eps);
    wn = __fsub_rn(wn, __fmul_rn(s.step_size, __fdiv_rn(mn, den)));
    w = wn;
    m = mn;
    v = vn;
    delta = __fsub_rn(wn, orig);
}

template <bool kPow2>
__device__ __forceinline__ void adamw_vec4(const StepScalars& s, const float4& a, float o0, float o1,
                                           float o2, float o3, float4& w, float4& m, float4& v,
                                           float4& d) {
    adamw_elem<kPow2>(s, a.x, o0, w.x, m.x, v.x, d.x);
    adamw_elem<kPow2>(s, a.y, o1, w.y, m.y, v.y, d.y);
    adamw_elem<kPow2>(s, a.z, o2, w.z, m.z, v.z, d.z);
    adamw_elem<kPow2>(s, a.w, o3, w.w, m.w, v.w, d.w);
}

// acc + (fp32)g for 8 elements, the same single fp32 add as the accumulate kernel.
__device__ __forceinline__ void add_grad8(float4& a0, float4& a1, const uint4& g) {
    a0.x = __fadd_rn(a0.x, bf16_lo(g.x));
    a0.y = __fadd_rn(a0.y, bf16_hi(g.x));
    a0.z = __fadd_rn(a0.z, bf16_lo(g.y));
    a0.w = __fadd_rn(a0.w, bf16_hi(g.y));
    a1.x = __fadd_rn(a1.x, bf16_lo(g.z));
    a1.y = __fadd_rn(a1.y, bf16_hi(g.z));
    a1.z = __fadd_rn(a1.z, bf16_lo(g.w));
    a1.w = __fadd_rn(a1.w, bf16_hi(g.w));
}

// One AdamW step over the chunk map.  In place: *_out == *_in (each element is
// read before it is written, by the same thread).  The accumulated grad sum is acc
// (+0.0 when acc is null) plus, when grad is set, the last micro-batch grad folded
// in here.  flags bit 0: reset acc to +0 afterwards.
// kSplit = 1: a CTA runs all kIters groups of its chunk; kSplit = kIters: kIters
// CTAs share a chunk, one group each (small launches: more, shorter CTAs fill the
// SMs in one wave instead of leaving a tail).
template <bool kPow2, int kSplit>
__device__ __forceinline__ void adamw_chunk(const StepDesc* __restrict__ dp, const Chunk c,
                                            const StepScalars& s) {
    const float* master_in = dp->master_in;
    const float* m_in = dp->m_in;
    const float* v_in = dp->v_in;
    float* acc = dp->acc;
    const uint16_t* orig = dp->orig;
    float* master_out = dp->master_out;
    float* m_out = dp->m_out;
    float* v_out = dp->v_out;
    float* delta = dp->delta;
    uint16_t* wbf = dp->w;
    const uint16_t* grad = dp->grad;
    const bool zero_acc = (dp->flags & kZeroAcc) != 0;
    const int64_t end = min(c.begin + kChunk, dp->n);

#pragma unroll 1
    for (int it = kSplit == 1 ? 0 : int(blockIdx.x % kSplit); it < kIters; it += kSplit) {
        const int64_t e = c.begin + (int64_t(it) * kThreads + threadIdx.x) * kVec;
        if (e + kVec <= end) {
            float4 w0 = ld_cs4(master_in + e), w1 = ld_cs4(master_in + e + 4);
            float4 m0 = ld_cs4(m_in + e), m1 = ld_cs4(m_in + e + 4);
            float4 v0 = ld_cs4(v_in + e), v1 = ld_cs4(v_in + e + 4);
            float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
            if (acc) {
                a0 = ld_cs4(acc + e);
                a1 = ld_cs4(acc + e + 4);
            }
            uint4 g = make_uint4(0u, 0u, 0u, 0u);
            if (grad) g = ld_cs8(grad + e);
            const uint4 o = ld_cs8(orig + e);
            if (grad) add_grad8(a0, a1, g);
            float4 d0, d1;
            adamw_vec4<kPow2>(s, a0, bf16_lo(o.x), bf16_hi(o.x), bf16_lo(o.y), bf16_hi(o.y),
                              w0, m0, v0, d0);
            adamw_vec4<kPow2>(s, a1, bf16_lo(o.z), bf16_hi(o.z), bf16_lo(o.w), bf16_hi(o.w),
                              w1, m1, v1, d1);
            st_cs4(master_out + e, w0);
            st_cs4(master_out + e + 4, w1);
            st_cs4(m_out + e, m0);
            st_cs4(m_out + e + 4, m1);
            st_cs4(v_out + e, v0);
            st_cs4(v_out + e + 4, v1);
            st_cs4(delta + e, d0);
            st_cs4(delta + e + 4, d1);
            uint4 wb;
            wb.x = bf16x2_rne(w0.x, w0.y);
            wb.y = bf16x2_rne(w0.z, w0.w);
            wb.z = bf16x2_rne(w1.x, w1.y);
            wb.w = bf16x2_rne(w1.z, w1.w);
            st_cs8(wbf + e, wb);
            if (zero_acc) {
                const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
                st_cs4(acc + e, z);
                st_cs4(acc + e + 4, z);
            }
        } else if (e < end) {
            // Ragged tail of the tensor (n not a multiple of 8): element by element.
            for (int64_t i = e; i < end; ++i) {
                float w = master_in[i], m = m_in[i], v = v_in[i], d;
                float a = acc ? acc[i] : 0.f;
                if (grad) a = __fadd_rn(a, bf16_one(grad + i));
                adamw_elem<kPow2>(s, a, bf16_one(orig + i), w, m, v, d);
                master_out[i] = w;
                m_out[i] = m;
                v_out[i] = v;
                delta[i] = d;
                wbf[i] = bf16_rne(w);
                if (zero_acc) acc[i] = 0.f;
            }
        }
    }
}

// Programmatic dependent launch.  The accumulate and step kernels may be launched
// with programmatic stream serialization, so that their CTAs are scheduled while
// the kernel before them on the stream drains (the launch latency of a small
// launch then overlaps that kernel's tail).  Each CTA first waits for the kernels
// it depends on to complete and their memory to be visible, before any global
// access, and then lets the next launch be scheduled.  Launched the plain way,
// both instructions return at once.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <bool kPow2, int kSplit>
__global__ void __launch_bounds__(kThreads)
adamw_fused_kernel(const StepDesc* __restrict__ descs, const Chunk* __restrict__ chunks,
                   const StepScalars s) {
    pdl_enter();
    const Chunk c = chunks[blockIdx.x / kSplit];
    adamw_chunk<kPow2, kSplit>(descs + c.tensor, c, s);
}

template <bool kPow2, int kSplit, int N>
__global__ void __launch_bounds__(kThreads)
adamw_fused_kernel_v(const __grid_constant__ DescTable<StepDesc, N> t,
                     const Chunk* __restrict__ chunks, const StepScalars s) {
    pdl_enter();
    const Chunk c = chunks[blockIdx.x / kSplit];
    adamw_chunk<kPow2, kSplit>(&t.d[c.tensor], c, s);
}

// acc_out = acc_in + (fp32)g, or +0.0 + (fp32)g when acc_in is null (the first
// micro-step; adding to +0.0 turns a -0 grad into +0, as the in-place form would).
template <int kSplit>   // as adamw_chunk
__device__ __forceinline__ void accum_chunk(const AccDesc* __restrict__ dp, const Chunk c) {
    const float* acc_in = dp->acc_in;
    float* acc_out = dp->acc_out;
    const uint16_t* grad = dp->grad;
    const int64_t end = min(c.begin + kChunk, dp->n);
    const bool from_zero = acc_in == nullptr;

#pragma unroll
    for (int it = kSplit == 1 ? 0 : int(blockIdx.x % kSplit); it < kIters; it += kSplit) {
        const int64_t e = c.begin + (int64_t(it) * kThreads + threadIdx.x) * kVec;
        if (e + kVec <= end) {
            const uint4 g = ld_cs8(grad + e);
            float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
            if (!from_zero) {
                a0 = ld_cs4(acc_in + e);
                a1 = ld_cs4(acc_in + e + 4);
            }
            add_grad8(a0, a1, g);
            st_cs4(acc_out + e, a0);
            st_cs4(acc_out + e + 4, a1);
        } else if (e < end) {
            for (int64_t i = e; i < end; ++i) {
                const float a = from_zero ? 0.f : acc_in[i];
                acc_out[i] = __fadd_rn(a, bf16_one(grad + i));
            }
        }
    }
}

template <int kSplit>
__global__ void __launch_bounds__(kThreads)
accum_grad_kernel(const AccDesc* __restrict__ descs, const Chunk* __restrict__ chunks) {
    pdl_enter();
    const Chunk c = chunks[blockIdx.x / kSplit];
    accum_chunk<kSplit>(descs + c.tensor, c);
}

template <int kSplit, int N>
__global__ void __launch_bounds__(kThreads)
accum_grad_kernel_v(const __grid_constant__ DescTable<AccDesc, N> t,
                    const Chunk* __restrict__ chunks) {
    pdl_enter();
    const Chunk c = chunks[blockIdx.x / kSplit];
    accum_chunk<kSplit>(&t.d[c.tensor], c);
}

// merged = bf16(base + delta): one fp32 add, round to nearest even (8 B/element:
// read bf16 2 + fp32 4, write bf16 2).
__global__ void __launch_bounds__(kThreads)
merge_kernel(const MergeDesc* __restrict__ descs, const Chunk* __restrict__ chunks) {
    const Chunk c = chunks[blockIdx.x];
    const MergeDesc* dp = descs + c.tensor;
    const uint16_t* base = dp->base;
    const float* delta = dp->delta;
    uint16_t* merged = dp->merged;
    const int64_t end = min(c.begin + kChunk, dp->n);
#pragma unroll
    for (int it = 0; it < kIters; ++it) {
        const int64_t e = c.begin + (int64_t(it) * kThreads + threadIdx.x) * kVec;
        if (e + kVec <= end) {
            const uint4 b = ld_cs8(base + e);
            const float4 d0 = ld_cs4(delta + e), d1 = ld_cs4(delta + e + 4);
            uint4 out;
            out.x = bf16x2_rne(__fadd_rn(bf16_lo(b.x), d0.x), __fadd_rn(bf16_hi(b.x), d0.y));
            out.y = bf16x2_rne(__fadd_rn(bf16_lo(b.y), d0.z), __fadd_rn(bf16_hi(b.y), d0.w));
            out.z = bf16x2_rne(__fadd_rn(bf16_lo(b.z), d1.x), __fadd_rn(bf16_hi(b.z), d1.y));
            out.w = bf16x2_rne(__fadd_rn(bf16_lo(b.w), d1.z), __fadd_rn(bf16_hi(b.w), d1.w));
            st_cs8(merged + e, out);
        } else if (e < end) {
            for (int64_t i = e; i < end; ++i)
                merged[i] = bf16_rne(__fadd_rn(bf16_one(base + i), delta[i]));
        }
    }
}

// Copy a descriptor table from pinned host memory (read through its unified
// address, volatile so no stale line is reused) into device memory.  The SMs do
// this copy so that it never queues behind bulk transfers on a copy engine.
__global__ void __launch_bounds__(kThreads)
install_table_kernel(uint4* __restrict__ dst, const uint4* __restrict__ src, int64_t n16) {
    for (int64_t i = int64_t(blockIdx.x) * kThreads + threadIdx.x; i < n16;
         i += int64_t(gridDim.x) * kThreads)
        dst[i] = __ldcv(src + i);
}

}  // namespace

cudaError_t launch_install(void* dst, const void* src, size_t bytes, cudaStream_t stream) {
    const int64_t n16 = int64_t(bytes / 16);
    if (n16 <= 0) return cudaSuccess;
    const unsigned blocks = unsigned(std::min<int64_t>((n16 + kThreads - 1) / kThreads, 1024));
    install_table_kernel<<<blocks, kThreads, 0, stream>>>(static_cast<uint4*>(dst),
                                                         static_cast<const uint4*>(src), n16);
    return cudaGetLastError();
}

// Launches of fewer chunks than this many per SM split each chunk over kIters CTAs.
constexpr int kSplitBelowChunksPerSm = 4;

// SM count of the current device, cached per device in a fixed table (no heap
// allocation: lema_adamw_step_noalloc launches through here too).
cudaError_t sm_count(int* out) {
    constexpr int kMaxDevices = 64;
    static std::mutex mu;
    static int cache[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> g(mu);
    if (cache[dev] == 0) {
        e = cudaDeviceGetAttribute(&cache[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    *out = cache[dev];
    return cudaSuccess;
}

cudaError_t split_launch(int64_t n_chunks, bool* split) {
    int sms = 0;
    const cudaError_t e = sm_count(&sms);
    if (e != cudaSuccess) return e;
    *split = n_chunks < int64_t(kSplitBelowChunksPerSm) * sms;
    return cudaSuccess;
}

namespace {

// One launch of kThreads-thread CTAs, with programmatic stream serialization when
// `pdl` (see pdl_enter).
template <typename... P, typename... A>
cudaError_t launch_k(void (*kernel)(P...), unsigned grid, cudaStream_t stream, bool pdl,
                     A... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace

cudaError_t launch_accum(const AccDesc* descs, const Chunk* chunks, int64_t n_chunks,
                         cudaStream_t stream, bool pdl) {
    if (n_chunks <= 0) return cudaSuccess;
    bool split = false;
    const cudaError_t e = split_launch(n_chunks, &split);
    if (e != cudaSuccess) return e;
    if (split)
        return launch_k(accum_grad_kernel<kIters>, unsigned(n_chunks * kIters), stream, pdl,
                        descs, chunks);
    return launch_k(accum_grad_kernel<1>, unsigned(n_chunks), stream, pdl, descs, chunks);
}

namespace {

template <typename D, int N>
DescTable<D, N> table_of(const D* host, int32_t count) {
    DescTable<D, N> t;
    std::memset(&t, 0, sizeof t);
    std::memcpy(t.d, host, sizeof(D) * size_t(count));
    return t;
}

template <int N>
cudaError_t accum_v(const AccDesc* host, int32_t count, const Chunk* chunks, int64_t n_chunks,
                    bool split, cudaStream_t stream, bool pdl) {
    const DescTable<AccDesc, N> t = table_of<AccDesc, N>(host, count);
    if (split)
        return launch_k(accum_grad_kernel_v<kIters, N>, unsigned(n_chunks * kIters), stream, pdl,
                        t, chunks);
    return launch_k(accum_grad_kernel_v<1, N>, unsigned(n_chunks), stream, pdl, t, chunks);
}

template <int N>
cudaError_t step_v(const StepDesc* host, int32_t count, const Chunk* chunks, int64_t n_chunks,
                   bool split, const StepScalars& s, cudaStream_t stream, bool pdl) {
    const DescTable<StepDesc, N> t = table_of<StepDesc, N>(host, count);
    const unsigned whole = unsigned(n_chunks), parts = unsigned(n_chunks * kIters);
    if (s.accum_pow2) {
        if (split) return launch_k(adamw_fused_kernel_v<true, kIters, N>, parts, stream, pdl, t, chunks, s);
        return launch_k(adamw_fused_kernel_v<true, 1, N>, whole, stream, pdl, t, chunks, s);
    }
    if (split) return launch_k(adamw_fused_kernel_v<false, kIters, N>, parts, stream, pdl, t, chunks, s);
    return launch_k(adamw_fused_kernel_v<false, 1, N>, whole, stream, pdl, t, chunks, s);
}

}  // namespace

cudaError_t launch_accum_v(const AccDesc* host_descs, int32_t count, const Chunk* chunks,
                           int64_t n_chunks, cudaStream_t stream, bool pdl) {
    if (n_chunks <= 0) return cudaSuccess;
    if (count > kValueTableMax) return cudaErrorInvalidValue;
    bool split = false;
    const cudaError_t e = split_launch(n_chunks, &split);
    if (e != cudaSuccess) return e;
    if (count <= kValueTableSmall)
        return accum_v<kValueTableSmall>(host_descs, count, chunks, n_chunks, split, stream, pdl);
    return accum_v<kValueTableMax>(host_descs, count, chunks, n_chunks, split, stream, pdl);
}

cudaError_t launch_step_v(const StepDesc* host_descs, int32_t count, const Chunk* chunks,
                          int64_t n_chunks, const StepScalars& s, cudaStream_t stream, bool pdl) {
    if (n_chunks <= 0) return cudaSuccess;
    if (count > kValueTableMax) return cudaErrorInvalidValue;
    bool split = false;
    const cudaError_t e = split_launch(n_chunks, &split);
    if (e != cudaSuccess) return e;
    if (count <= kValueTableSmall)
        return step_v<kValueTableSmall>(host_descs, count, chunks, n_chunks, split, s, stream, pdl);
    return step_v<kValueTableMax>(host_descs, count, chunks, n_chunks, split, s, stream, pdl);
}

cudaError_t launch_merge(const MergeDesc* descs, const Chunk* chunks, int64_t n_chunks,
                         cudaStream_t stream) {
    if (n_chunks <= 0) return cudaSuccess;
    merge_kernel<<<dim3(unsigned(n_chunks)), kThreads, 0, stream>>>(descs, chunks);
    return cudaGetLastError();
}


cudaError_t launch_step(const StepDesc* descs, const Chunk* chunks, int64_t n_chunks,
                        const StepScalars& s, cudaStream_t stream, bool pdl) {
    if (n_chunks <= 0) return cudaSuccess;
    bool split = false;
    const cudaError_t e = split_launch(n_chunks, &split);
    if (e != cudaSuccess) return e;
    const unsigned whole = unsigned(n_chunks), parts = unsigned(n_chunks * kIters);
    if (s.accum_pow2) {
        if (split) return launch_k(adamw_fused_kernel<true, kIters>, parts, stream, pdl, descs, chunks, s);
        return launch_k(adamw_fused_kernel<true, 1>, whole, stream, pdl, descs, chunks, s);
    }
    if (split) return launch_k(adamw_fused_kernel<false, kIters>, parts, stream, pdl, descs, chunks, s);
    return launch_k(adamw_fused_kernel<false, 1>, whole, stream, pdl, descs, chunks, s);
}

}  // namespace lema
