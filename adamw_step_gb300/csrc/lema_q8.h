// lema_q8.h -- descriptors and entry points of the 8-bit-state kernels of
// liblema.so (lema_kernels_q8.cu; not part of the public ABI).
#pragma once

#include "lema_internal.h"

namespace lema {

// 8-bit states: blocks of kQBlock consecutive elements share one fp32 scale; one
// warp (32 lanes x kVec elements) covers exactly one block.
constexpr int kQBlock = 256;
static_assert(kQBlock == 32 * kVec, "a warp covers one quantization block");

// Step descriptor, 8-bit moments (m as int8, sqrt(v) as uint8) and accumulator.
// In place: the *_out pointers equal the inputs.  acc_q may be null (K = 1 with
// grad); flags bit 0 (kZeroAcc): reset the accumulator's codes and scales to 0.
struct alignas(16) StepDescQ8 {
    const float* master_in;
    const int8_t* m_q_in;
    const float* m_scale_in;
    const uint8_t* r_q_in;
    const float* r_scale_in;
    int8_t* acc_q;
    float* acc_scale;
    const uint16_t* grad;
    const uint16_t* orig;
    float* master_out;
    int8_t* m_q_out;
    float* m_scale_out;
    uint8_t* r_q_out;
    float* r_scale_out;
    float* delta;
    uint16_t* w;
    int64_t n;
    int64_t flags;
};
static_assert(sizeof(StepDescQ8) == 144, "StepDescQ8 layout");

// Accumulate descriptor, 8-bit accumulator: out = encode(decode(in) + g), or
// encode(+0 + g) when acc_q_in is null.
struct alignas(16) AccDescQ8 {
    const int8_t* acc_q_in;
    const float* acc_scale_in;
    int8_t* acc_q_out;
    float* acc_scale_out;
    const uint16_t* grad;
    int64_t n;
};
static_assert(sizeof(AccDescQ8) == 48, "AccDescQ8 layout");

// Kernel launchers (lema_kernels_q8.cu).  `descs` and `chunks` are device tables.
cudaError_t launch_accum_q8(const AccDescQ8* descs, const Chunk* chunks, int64_t n_chunks,
                            cudaStream_t stream);
// gave_up: device-visible address of a word in host-mapped memory that the kernel
// sets to 1 when one of its bounded waits runs out (may be null).
cudaError_t launch_step_q8(const StepDescQ8* descs, const Chunk* chunks, int64_t n_chunks,
                           const StepScalars& s, unsigned int* gave_up, cudaStream_t stream);

// By-value descriptor tables (at most kValueTableMax tensors), as launch_step_v.
cudaError_t launch_accum_q8_v(const AccDescQ8* host_descs, int32_t count, const Chunk* chunks,
                              int64_t n_chunks, cudaStream_t stream);
cudaError_t launch_step_q8_v(const StepDescQ8* host_descs, int32_t count, const Chunk* chunks,
                             int64_t n_chunks, const StepScalars& s, unsigned int* gave_up,
                             cudaStream_t stream);

// Count of kernel-side bounded waits (the staged 8-bit step's mbarrier waits) that
// ran out since the library was loaded on this device.
cudaError_t read_wait_timeouts(unsigned long long* out);
// Test: every x >= 0 through the 8-bit step's division by a per-call constant
// against the IEEE division; adds the mismatches inside (bad_dev[0]) and outside
// (bad_dev[1]) its domain.
cudaError_t check_div_by_const(float c, float rc, unsigned long long* bad_dev,
                               cudaStream_t stream);
// The staged 8-bit step's wait limit on the current device (ns < 0: the default).
cudaError_t set_wait_limit(int64_t ns);

// A word of host-mapped, page-locked memory that an 8-bit step kernel sets when a
// bounded wait runs out: `host` is read by the library after the work has finished,
// `dev` is the address passed to the kernel.
struct GaveUpFlag {
    volatile unsigned int* host = nullptr;
    unsigned int* dev = nullptr;
};
int gave_up_flag_alloc(GaveUpFlag* f);
void gave_up_flag_free(GaveUpFlag* f);
// LEMA_ERR_TIMEOUT (and the flag cleared) when the flag is set, else LEMA_OK.
int gave_up_take(const GaveUpFlag& f, const char* where);

// Validate + build-or-reuse the device table + launch (lema_api.cu).
int run_accum_q8(const AccDescQ8* descs, int32_t count, cudaStream_t stream);
int run_step_q8(const StepDescQ8* descs, int32_t count, const StepScalars& s, cudaStream_t stream,
                unsigned int* gave_up);

}  // namespace lema
