// lema_internal.h -- shapes shared by the host library and the kernels of
// liblema.so (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "lema.h"

namespace lema {

// Work decomposition: a launch covers a list of 1-D tensors; each tensor is cut
// into chunks of kChunk elements (the last one ragged) and each CTA of kThreads
// threads owns one chunk.  A thread moves kVec consecutive elements per iteration
// (16-byte accesses: 2 x float4 per fp32 stream, 1 x uint4 per bf16 stream).
constexpr int kThreads = 256;
constexpr int kVec = 8;
constexpr int kIters = 4;
constexpr int64_t kChunk = int64_t(kThreads) * kVec * kIters;  // 8192 elements

// One entry of the step's device-side descriptor table.  In place: *_out == the
// input pointer.  The accumulated sum is acc (or +0.0 when acc is null) plus, when
// grad is set, the folded-in last micro-batch grad.  flags bit 0 (kZeroAcc): reset
// acc to +0.0 after reading it (the public in-place step); out-of-place steps leave
// every input untouched.
struct alignas(16) StepDesc {
    const float* master_in;
    const float* m_in;
    const float* v_in;
    float* acc;
    const uint16_t* orig;
    float* master_out;
    float* m_out;
    float* v_out;
    float* delta;
    uint16_t* w;
    const uint16_t* grad;
    int64_t n;
    int64_t flags;      // bit 0 = kZeroAcc
};
static_assert(sizeof(StepDesc) == 112, "StepDesc layout");
constexpr int64_t kZeroAcc = 1;

// One entry of the accumulate kernel's table: acc_out = (acc_in or +0) + g.
struct alignas(16) AccDesc {
    const float* acc_in;   // nullptr: start from +0.0 (first micro-step)
    float* acc_out;        // == acc_in for the in-place public entry point
    const uint16_t* grad;
    int64_t n;
};
static_assert(sizeof(AccDesc) == 32, "AccDesc layout");

// Chunk map entry: chunk [begin, min(begin + kChunk, n)) of tensor `tensor`.
struct alignas(16) Chunk {
    int32_t tensor;
    int32_t reserved;
    int64_t begin;
};
static_assert(sizeof(Chunk) == 16, "Chunk layout");

// Merge descriptor: merged = bf16(base + delta); merged may be base (in place).
struct alignas(16) MergeDesc {
    const uint16_t* base;
    const float* delta;
    uint16_t* merged;
    int64_t n;
};
static_assert(sizeof(MergeDesc) == 32, "MergeDesc layout");

// Per-call fp32 scalars (formed on the host in fp64, rounded once).
struct StepScalars {
    float decay;       // 1 - lr*wd
    float beta1;
    float omb1;        // 1 - beta1
    float beta2;
    float omb2;        // 1 - beta2
    float step_size;   // lr / (1 - beta1^t)
    float bc2_sqrt;    // sqrt(1 - beta2^t)
    float eps;
    float accum;       // K
    float inv_accum;   // 1/K, exact when K is a power of two
    float bc2_rcp;     // 1 / bc2_sqrt, correctly rounded (rcp_rn)
    int32_t accum_pow2;
};

// Kernel launchers (lema_kernels.cu; the 8-bit ones are declared in lema_q8.h).
// `descs` and `chunks` are device tables.
// pdl: launch with programmatic stream serialization (the kernel is scheduled while
// the one before it on the stream drains, and waits for it before any memory access).
cudaError_t launch_accum(const AccDesc* descs, const Chunk* chunks, int64_t n_chunks,
                         cudaStream_t stream, bool pdl = false);
cudaError_t launch_step(const StepDesc* descs, const Chunk* chunks, int64_t n_chunks,
                        const StepScalars& s, cudaStream_t stream, bool pdl = false);
cudaError_t launch_merge(const MergeDesc* descs, const Chunk* chunks, int64_t n_chunks,
                         cudaStream_t stream);
// A descriptor table of up to N tensors passed by value as a kernel parameter
// (__grid_constant__): a call is then one launch, with no table upload.
template <typename D, int N>
struct DescTable {
    D d[N];
};

// The same kernels with the descriptor table passed by value as a kernel parameter
// (`host_descs` is read on the host at launch; at most kValueTableMax tensors), so
// a call needs no table upload.
constexpr int kValueTableSmall = 16;   // 16 x 112 B = 1.8 KB of parameters
constexpr int kValueTableMax = 64;     // 64 x 112 B = 7.2 KB
cudaError_t launch_accum_v(const AccDesc* host_descs, int32_t count, const Chunk* chunks,
                           int64_t n_chunks, cudaStream_t stream, bool pdl = false);
cudaError_t launch_step_v(const StepDesc* host_descs, int32_t count, const Chunk* chunks,
                          int64_t n_chunks, const StepScalars& s, cudaStream_t stream,
                          bool pdl = false);
// SM-driven copy of `bytes` (a multiple of 16) from pinned host to device memory.
cudaError_t launch_install(void* dst, const void* src, size_t bytes, cudaStream_t stream);

// Host library helpers (lema_api.cu), also used by the pool.
int set_error(int status, const char* fmt, ...);
void clear_error();
int cuda_error(cudaError_t e, const char* what);
int make_scalars(int64_t step, double lr, double beta1, double beta2, double eps,
                 double weight_decay, int32_t accum_steps, StepScalars* out);
// The fp32 reciprocal of a positive normal c, correctly rounded (RN(1/c)).
float rcp_rn(float c);
// Validate + build-or-reuse the device table + launch.  Host arrays of descriptors.
// pdl: as the launchers' (the public resident entry points pass true).
int run_accum(const AccDesc* descs, int32_t count, cudaStream_t stream, bool pdl = false);
int run_step(const StepDesc* descs, int32_t count, const StepScalars& s, cudaStream_t stream,
             bool pdl = false);
int run_merge(const MergeDesc* descs, int32_t count, cudaStream_t stream);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace lema
