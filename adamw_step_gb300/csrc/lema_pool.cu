// lema_pool.cu -- streamed residency: fp32 optimizer states in pinned host RAM,
// moved layer by layer through a pool of VRAM slots on three CUDA streams.
//
// Page "LEMA: Layer-wise Efficient Memory Abstraction": section "Features" (pinned
// RAM -> VRAM with asynchronous prefetch hides the host link; a sliding-window pool
// keeps VRAM constant whatever the depth; fp32 optimizer states virtualised into
// RAM like the weights) and section "TensorStore: Unified Streaming Core" (one
// slot-pool address space for weights, optimizer states and gradient accumulators,
// with a residency policy per stream).  The pages' disk tier and triple buffer are
// prior art; here the unit of streaming is one layer (or the embedding / head),
// and the copy engines do the moving while the SMs run the step.
//
// Slot layout (P = slot capacity in elements, padded to 128):
//   input half : master, m, v, acc (fp32, 4P each), orig, grad (bf16, 2P each)
//   output half: master', m', v', delta (fp32, 4P each), w (bf16, 2P)
// The accumulate-only micro-steps write acc' into the output half's delta region,
// so the next unit's host-to-device copy into a slot's input half never races the
// device-to-host copy out of its output half.
//
// A unit laid out packed (LEMA_UNIT_PACKED) can be moved in up to kMaxSlices slices
// of whole chunks (lema_pool_slices; whole units by default): slice q's
// host-to-device copies, its kernel and its device-to-host copies each start as
// soon as slice q of the stage before is done, so a unit's kernel starts after one
// slice has arrived instead of the whole unit.  Measured, that does not shorten the
// streamed steps: their last micro-step sends more bytes to the host than it reads
// from it, so that tail stays, and with the directions overlapping more each runs
// slower.
//
// Ordering (per slot s, per unit L, per slice q):
//   H2D(L, q)  (from q = 0: waits step_done[s], the input half free, and the D2H
//              events that last wrote the host buffers it reads); records in_ready[s][q].
//   step(L, q) (from q = 0: waits out_drained[s], the output half free); waits
//              in_ready[s][q]; records done[s][q]; after the last slice step_done[s].
//   D2H(L, q)  waits done[s][q]; after the last slice records out_drained[s] and
//              unit_done[L].
// Every wait is a device-side stream wait; the host never blocks inside a call.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <mutex>
#include <thread>
#include <unordered_map>
#include <vector>

#include "lema_internal.h"
#include "lema_pool_impl.h"
#include "lema_q8.h"

using namespace lema;

namespace {

constexpr int kMaxSlices = 8;             // slices of one unit (see lema_pool_slices)
constexpr int64_t kSliceAlign = kChunk;    // slice boundaries: whole chunks

struct Slot {
    float* master = nullptr;
    float* m = nullptr;
    float* v = nullptr;
    float* acc = nullptr;
    uint16_t* orig = nullptr;
    uint16_t* grad = nullptr;
    float* master_o = nullptr;
    float* m_o = nullptr;
    float* v_o = nullptr;
    float* delta = nullptr;
    uint16_t* w = nullptr;
    cudaEvent_t in_ready[kMaxSlices] = {}, done[kMaxSlices] = {};
    cudaEvent_t step_done = nullptr, out_drained = nullptr;
};

constexpr int64_t kTensorAlign = 64;  // elements; keeps every sub-array 128-byte aligned

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

std::atomic<int64_t> g_fail_copy{0};

int copy_async(void* dst, const void* src, int64_t bytes, cudaMemcpyKind kind, cudaStream_t s) {
    if (bytes <= 0) return LEMA_OK;
    int64_t k = g_fail_copy.load();
    while (k > 0 && !g_fail_copy.compare_exchange_weak(k, k - 1)) {}
    if (k == 1) return set_error(LEMA_ERR_CUDA, "injected host<->device copy failure (test hook)");
    cudaError_t e = cudaMemcpyAsync(dst, src, size_t(bytes), kind, s);
    return e == cudaSuccess ? LEMA_OK : cuda_error(e, "cudaMemcpyAsync");
}

int wait_on(cudaStream_t s, cudaEvent_t ev) {
    cudaError_t e = cudaStreamWaitEvent(s, ev, 0);
    return e == cudaSuccess ? LEMA_OK : cuda_error(e, "cudaStreamWaitEvent");
}

int record(cudaEvent_t ev, cudaStream_t s) {
    cudaError_t e = cudaEventRecord(ev, s);
    return e == cudaSuccess ? LEMA_OK : cuda_error(e, "cudaEventRecord");
}

// 1 = pinned host, 2 = memory of the current device (or managed), 0 = anything else
// (pageable host memory, another GPU's memory).
int memory_kind(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (a.type == cudaMemoryTypeHost) return 1;
    if (a.type == cudaMemoryTypeManaged) return 2;
    if (a.type == cudaMemoryTypeDevice) {
        int dev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        return a.device == dev ? 2 : 0;
    }
    return 0;
}

#define LEMA_TRY(expr)                       \
    do {                                     \
        int rc_ = (expr);                    \
        if (rc_ != LEMA_OK) return rc_;      \
    } while (0)

}  // namespace

struct lema_pool {
    int device = 0;
    int n_slots = 0;
    int64_t slot_params = 0;
    int64_t slot_bytes = 0;
    void* slab = nullptr;
    std::vector<Slot> slots;
    cudaStream_t h2d = nullptr, cmp = nullptr, d2h = nullptr;
    cudaEvent_t entry = nullptr;
    cudaEvent_t tail[3] = {nullptr, nullptr, nullptr};
    std::vector<cudaEvent_t> unit_done;                   // per unit index of a call
    std::unordered_map<const void*, size_t> last_writer;  // host buffer -> unit_done index
    std::unordered_map<const void*, int> kinds;            // memory_kind() of checked pointers
    int64_t next_slot = 0;
    GaveUpFlag gave_up;   // set by an 8-bit step kernel of this pool whose wait ran out
    bool copies_only = false;   // measurement mode: no kernels (lema_pool_copies_only)
    int32_t max_slices = 1;                   // lema_pool_slices (default: whole units)
    bool slice_first_only = false;            // lema_pool_slice_first_unit
    int64_t min_slice = int64_t(8) << 20;     // elements
    std::mutex mu;
    // Stage tracing (off unless lema_pool_trace enabled it): a timed event pair per
    // stage of each unit, recorded on the stage's stream after its waits.
    struct TraceRec {
        int32_t stage, unit, call;
        cudaEvent_t start, end;
    };
    std::vector<TraceRec> trace;
    int32_t trace_cap = 0;
    int32_t calls = 0;
};

namespace {

void clear_trace(lema_pool* p) {
    for (auto& r : p->trace) {
        cudaEventDestroy(r.start);
        cudaEventDestroy(r.end);
    }
    p->trace.clear();
}

// Open a traced stage on stream s (no-op unless tracing is on and has room).
int trace_open(lema_pool* p, cudaStream_t s, int32_t stage, int32_t unit, int* idx) {
    *idx = -1;
    if (int32_t(p->trace.size()) >= p->trace_cap) return LEMA_OK;
    lema_pool::TraceRec r{stage, unit, p->calls, nullptr, nullptr};
    cudaError_t e = cudaEventCreate(&r.start);
    if (e == cudaSuccess) e = cudaEventCreate(&r.end);
    if (e == cudaSuccess) e = cudaEventRecord(r.start, s);
    if (e != cudaSuccess) return cuda_error(e, "trace event");
    *idx = int(p->trace.size());
    p->trace.push_back(r);
    return LEMA_OK;
}

int trace_close(lema_pool* p, cudaStream_t s, int idx) {
    if (idx < 0) return LEMA_OK;
    cudaError_t e = cudaEventRecord(p->trace[size_t(idx)].end, s);
    return e == cudaSuccess ? LEMA_OK : cuda_error(e, "trace event");
}

void destroy_pool(lema_pool* p) {
    if (p->h2d) cudaStreamSynchronize(p->h2d);
    if (p->cmp) cudaStreamSynchronize(p->cmp);
    if (p->d2h) cudaStreamSynchronize(p->d2h);
    clear_trace(p);
    for (Slot& s : p->slots) {
        for (int q = 0; q < kMaxSlices; ++q) {
            if (s.in_ready[q]) cudaEventDestroy(s.in_ready[q]);
            if (s.done[q]) cudaEventDestroy(s.done[q]);
        }
        if (s.step_done) cudaEventDestroy(s.step_done);
        if (s.out_drained) cudaEventDestroy(s.out_drained);
    }
    for (cudaEvent_t e : p->unit_done) cudaEventDestroy(e);
    for (cudaEvent_t e : p->tail)
        if (e) cudaEventDestroy(e);
    if (p->entry) cudaEventDestroy(p->entry);
    if (p->h2d) cudaStreamDestroy(p->h2d);
    if (p->cmp) cudaStreamDestroy(p->cmp);
    if (p->d2h) cudaStreamDestroy(p->d2h);
    if (p->slab) cudaFree(p->slab);
    gave_up_flag_free(&p->gave_up);
    delete p;
}

int new_event(cudaEvent_t* e) {
    cudaError_t r = cudaEventCreateWithFlags(e, cudaEventDisableTiming);
    return r == cudaSuccess ? LEMA_OK : cuda_error(r, "cudaEventCreate");
}

// The slices of a unit whose packed span holds n_span elements: S pieces, bound[0]
// = 0 < bound[1] < ... < bound[S] = n_span, inner boundaries on whole chunks, each
// piece at least the pool's minimum slice; S = 1 for a unit that is not packed, and
// for every unit but the call's first (slot-using) one when the pool slices only that.
int unit_slices(const lema_pool* p, bool packed, bool first_unit, int64_t n_span,
                int64_t* bound) {
    bound[0] = 0;
    const bool sliced = packed && (first_unit || !p->slice_first_only);
    int64_t want = sliced ? std::min<int64_t>(p->max_slices, n_span / p->min_slice) : 1;
    want = std::max<int64_t>(1, std::min<int64_t>(want, kMaxSlices));
    int S = 0;
    for (int64_t q = 1; q < want; ++q) {
        const int64_t b = round_up(n_span * q / want, kSliceAlign);
        if (b > bound[S] && b < n_span) bound[++S] = b;
    }
    bound[++S] = n_span;
    return S;
}

// memory_kind() once per pointer per pool: the driver's lookup grows with the number
// of registered host ranges, and a whole model passes thousands of buffers per call.
// Only pinned and device answers are kept: a buffer rejected now may be registered
// and passed again.  The cache is emptied when it grows past kMaxKinds entries (a
// caller passing fresh buffers every call).
int cached_kind(std::unordered_map<const void*, int>& cache, const void* p) {
    constexpr size_t kMaxKinds = size_t(1) << 20;
    auto it = cache.find(p);
    if (it != cache.end()) return it->second;
    const int k = memory_kind(p);
    if (k != 0) {
        if (cache.size() >= kMaxKinds) cache.clear();
        cache.emplace(p, k);
    }
    return k;
}

// The writer map orders each host buffer's next read after the device-to-host copy
// that last wrote it.  It grows with the distinct host buffers a caller passes; past
// kMaxWriters entries it is emptied, which is safe once every copy the pool has
// enqueued on its device-to-host stream is done: wait for that (bounded) first.
int bound_writers(lema_pool* pool);
int begin_call(lema_pool* pool, int32_t n_units, cudaStream_t caller);
void note_writer(lema_pool* pool, const void* p, std::vector<size_t>& waits);
int wait_for_writers(lema_pool* pool, std::vector<size_t>& waits);
int end_call(lema_pool* pool);

// The residency of a unit's accumulators: every non-empty tensor's accumulator
// buffers (fp32: acc; 8-bit: codes and scales) in pinned host memory (1) or all in
// device memory (2).  *kind is 0 on entry and stays 0 for a unit with no data.
int check_acc_kind(const void* const* bufs, int n_bufs, int32_t L, int32_t j,
                   std::unordered_map<const void*, int>& kinds, int* kind) {
    for (int i = 0; i < n_bufs; ++i) {
        const void* p = bufs[i];
        if (!p) return set_error(LEMA_ERR_ARG, "unit %d tensor %d: NULL accumulator", L, j);
        if (!aligned16(p))
            return set_error(LEMA_ERR_ALIGN, "unit %d tensor %d: accumulator not 16-byte aligned",
                             L, j);
        const int k = cached_kind(kinds, p);
        if (k == 0)
            return set_error(LEMA_ERR_ARG,
                             "unit %d tensor %d: accumulator must be pinned host memory or memory "
                             "of the pool's GPU", L, j);
        if (*kind != 0 && k != *kind)
            return set_error(LEMA_ERR_ARG,
                             "unit %d tensor %d: a unit's accumulators must all be pinned host "
                             "memory or all device memory", L, j);
        *kind = k;
    }
    return LEMA_OK;
}

// Host-side checks of one unit for a streamed call; fills grad_on_host per tensor
// and *acc_on_device (the unit's accumulators live in device memory).
int check_streamed_unit(const lema_layer& ly, int32_t L, int32_t k, bool final_step,
                        int64_t slot_params, std::vector<char>& grad_on_host,
                        std::unordered_map<const void*, int>& kinds, bool* acc_on_device) {
    int64_t need = 0;
    int acc_kind = 0;
    for (int32_t j = 0; j < ly.count; ++j) {
        const lema_tensor& t = ly.tensors[j];
        if (t.n < 0) return set_error(LEMA_ERR_ARG, "unit %d tensor %d: n must be >= 0", L, j);
        need += round_up(t.n, kTensorAlign);
        grad_on_host.push_back(0);
        if (t.n == 0) continue;
        const int outs = (t.master_out != nullptr) + (t.m_out != nullptr) + (t.v_out != nullptr);
        if (outs != 0 && outs != 3)
            return set_error(LEMA_ERR_ARG,
                             "unit %d tensor %d: master_out, m_out, v_out must be all NULL or all set",
                             L, j);
        const void* acc[] = {t.acc};
        LEMA_TRY(check_acc_kind(acc, 1, L, j, kinds, &acc_kind));
        std::vector<const void*> host;
        if (final_step) {
            host.insert(host.end(), {t.master, t.m, t.v, t.orig_bf16, t.delta, t.w_bf16});
            if (outs) host.insert(host.end(), {t.master_out, t.m_out, t.v_out});
        }
        for (const void* p : host) {
            if (!p) return set_error(LEMA_ERR_ARG, "unit %d tensor %d: NULL host buffer", L, j);
            if (!aligned16(p))
                return set_error(LEMA_ERR_ALIGN, "unit %d tensor %d: host buffer not 16-byte aligned",
                                 L, j);
            if (cached_kind(kinds, p) != 1)
                return set_error(LEMA_ERR_ARG,
                                 "unit %d tensor %d: state buffers must be pinned host memory", L, j);
        }
        const uint16_t* g = ly.grads[j];
        if (!g) return set_error(LEMA_ERR_ARG, "unit %d tensor %d: NULL grad", L, j);
        if (!aligned16(g))
            return set_error(LEMA_ERR_ALIGN, "unit %d tensor %d: grad not 16-byte aligned", L, j);
        const int kind = cached_kind(kinds, g);
        if (kind == 0)
            return set_error(LEMA_ERR_ARG,
                             "unit %d tensor %d: grad must be memory of the pool's GPU or pinned "
                             "host memory", L, j);
        grad_on_host.back() = (kind == 1);
    }
    (void)k;
    *acc_on_device = acc_kind == 2;
    if (need > slot_params)
        return set_error(LEMA_ERR_ARG, "unit %d needs %lld slot elements, a slot holds %lld", L,
                         (long long)need, (long long)slot_params);
    if (ly.flags & ~int32_t(LEMA_UNIT_PACKED))
        return set_error(LEMA_ERR_ARG, "unit %d: unknown flags", L);
    if (ly.flags & LEMA_UNIT_PACKED) {
        // Every field of every non-empty tensor j must sit (o_j - o_first) elements
        // after the first non-empty tensor's (empty tensors carry no data and may
        // have any pointers).
        int32_t first = -1;
        int64_t o = 0, o_first = 0;
        for (int32_t j = 0; j < ly.count; ++j) {
            const lema_tensor& t = ly.tensors[j];
            const int64_t oj = o;
            o += round_up(t.n, kTensorAlign);
            if (t.n == 0) continue;
            if (first < 0) {
                first = j;
                o_first = oj;
            }
            const lema_tensor& t0 = ly.tensors[first];
            auto at = [&](const void* base, const void* p, int64_t size) {
                return reinterpret_cast<uintptr_t>(p) ==
                       reinterpret_cast<uintptr_t>(base) + uintptr_t((oj - o_first) * size);
            };
            // Only the fields this micro-step moves: acc (unless it stays in device
            // memory), and at the last micro-step the optimizer states and outputs.
            bool ok = *acc_on_device || at(t0.acc, t.acc, 4);
            if (final_step) {
                ok = ok && at(t0.master, t.master, 4) && at(t0.m, t.m, 4) && at(t0.v, t.v, 4) &&
                     at(t0.delta, t.delta, 4) && at(t0.orig_bf16, t.orig_bf16, 2) &&
                     at(t0.w_bf16, t.w_bf16, 2);
                if (t0.master_out)
                    ok = ok && at(t0.master_out, t.master_out, 4) && at(t0.m_out, t.m_out, 4) &&
                         at(t0.v_out, t.v_out, 4);
            }
            if (!ok)
                return set_error(LEMA_ERR_ARG,
                                 "unit %d is flagged packed but tensor %d is not at its slot offset",
                                 L, j);
        }
    }
    return LEMA_OK;
}

}  // namespace

namespace {
int64_t carved_q8_bytes(int64_t P);   // the 8-bit slot layout (below)
}  // namespace

// =================================================================== C ABI ====

extern "C" int lema_pool_create(int32_t n_slots, int64_t slot_params, lema_pool** out) {
    clear_error();
    if (!out) return set_error(LEMA_ERR_ARG, "out is NULL");
    *out = nullptr;
    if (n_slots < 2) return set_error(LEMA_ERR_ARG, "a pool needs at least 2 slots (got %d)", n_slots);
    if (slot_params < 1) return set_error(LEMA_ERR_ARG, "slot_params must be >= 1");
    lema_pool* p = new lema_pool();
    cudaError_t e = cudaGetDevice(&p->device);
    if (e != cudaSuccess) { destroy_pool(p); return cuda_error(e, "cudaGetDevice"); }
    p->n_slots = n_slots;
    p->slot_params = round_up(slot_params, 128);
    const int64_t P = p->slot_params;
    // 38 bytes per element hold the fp32 layout; the 8-bit carving (its fields each
    // rounded up to 256 bytes) needs a little more than its 24 bytes per element,
    // which only tiny slots notice.
    const size_t slot_bytes = size_t(std::max<int64_t>(P * 38, carved_q8_bytes(P)));
    p->slot_bytes = int64_t(slot_bytes);
    e = cudaMalloc(&p->slab, slot_bytes * size_t(n_slots));
    if (e != cudaSuccess) {
        p->slab = nullptr;
        destroy_pool(p);
        return set_error(LEMA_ERR_OOM, "slot pool of %d x %lld elements: %s", n_slots,
                         (long long)P, cudaGetErrorString(e));
    }
    p->slots.resize(size_t(n_slots));
    for (int i = 0; i < n_slots; ++i) {
        unsigned char* b = static_cast<unsigned char*>(p->slab) + slot_bytes * size_t(i);
        Slot& s = p->slots[size_t(i)];
        auto f32 = [&](float*& dst) { dst = reinterpret_cast<float*>(b); b += 4 * P; };
        auto b16 = [&](uint16_t*& dst) { dst = reinterpret_cast<uint16_t*>(b); b += 2 * P; };
        f32(s.master); f32(s.m); f32(s.v); f32(s.acc); b16(s.orig); b16(s.grad);
        f32(s.master_o); f32(s.m_o); f32(s.v_o); f32(s.delta); b16(s.w);
        int rc = new_event(&s.step_done);
        if (rc == LEMA_OK) rc = new_event(&s.out_drained);
        for (int q = 0; q < kMaxSlices && rc == LEMA_OK; ++q) {
            rc = new_event(&s.in_ready[q]);
            if (rc == LEMA_OK) rc = new_event(&s.done[q]);
        }
        if (rc != LEMA_OK) {
            destroy_pool(p);
            return rc;
        }
    }
    int rc;
    if ((rc = gave_up_flag_alloc(&p->gave_up)) != LEMA_OK) {
        destroy_pool(p);
        return rc;
    }
    if ((rc = new_event(&p->entry)) || (rc = new_event(&p->tail[0])) ||
        (rc = new_event(&p->tail[1])) || (rc = new_event(&p->tail[2]))) {
        destroy_pool(p);
        return rc;
    }
    if ((e = cudaStreamCreateWithFlags(&p->h2d, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&p->cmp, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&p->d2h, cudaStreamNonBlocking)) != cudaSuccess) {
        destroy_pool(p);
        return cuda_error(e, "cudaStreamCreate");
    }
    *out = p;
    return LEMA_OK;
}

extern "C" int lema_pool_destroy(lema_pool* pool) {
    clear_error();
    if (!pool) return LEMA_OK;
    destroy_pool(pool);
    return LEMA_OK;
}

extern "C" int lema_pool_sync(lema_pool* pool, int32_t timeout_ms) {
    clear_error();
    if (!pool) return set_error(LEMA_ERR_ARG, "pool is NULL");
    if (timeout_ms < 0) return set_error(LEMA_ERR_ARG, "timeout_ms must be >= 0");
    const auto deadline = std::chrono::steady_clock::now() + std::chrono::milliseconds(timeout_ms);
    for (;;) {
        bool pending = false;
        for (cudaEvent_t ev : pool->tail) {
            cudaError_t e = cudaEventQuery(ev);
            if (e == cudaErrorNotReady) { pending = true; continue; }
            if (e != cudaSuccess) return cuda_error(e, "pool work failed");
        }
        if (!pending) return gave_up_take(pool->gave_up, "lema_pool_sync");
        if (std::chrono::steady_clock::now() >= deadline)
            return set_error(LEMA_ERR_TIMEOUT, "pool work still pending after %d ms", timeout_ms);
        std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
}

extern "C" int lema_pool_wait_stream(lema_pool* pool, void* cuda_stream) {
    clear_error();
    if (!pool) return set_error(LEMA_ERR_ARG, "pool is NULL");
    for (cudaEvent_t ev : pool->tail) LEMA_TRY(wait_on(static_cast<cudaStream_t>(cuda_stream), ev));
    return LEMA_OK;
}

extern "C" int lema_pool_slices(lema_pool* pool, int32_t max_slices, int64_t min_slice_params) {
    clear_error();
    if (!pool) return set_error(LEMA_ERR_ARG, "pool is NULL");
    if (max_slices < 1 || max_slices > kMaxSlices)
        return set_error(LEMA_ERR_ARG, "max_slices must lie in [1, %d] (got %d)", kMaxSlices,
                         max_slices);
    if (min_slice_params < 1) return set_error(LEMA_ERR_ARG, "min_slice_params must be >= 1");
    std::lock_guard<std::mutex> lock(pool->mu);
    pool->max_slices = max_slices;
    pool->min_slice = round_up(min_slice_params, kSliceAlign);
    return LEMA_OK;
}

extern "C" int lema_pool_slice_first_unit(lema_pool* pool, int32_t on) {
    clear_error();
    if (!pool) return set_error(LEMA_ERR_ARG, "pool is NULL");
    std::lock_guard<std::mutex> lock(pool->mu);
    pool->slice_first_only = on != 0;
    return LEMA_OK;
}

extern "C" int lema_pool_copies_only(lema_pool* pool, int32_t on) {
    clear_error();
    if (!pool) return set_error(LEMA_ERR_ARG, "pool is NULL");
    std::lock_guard<std::mutex> lock(pool->mu);
    LEMA_TRY(lema_pool_sync(pool, 600000));
    pool->copies_only = on != 0;
    return LEMA_OK;
}

extern "C" void lema_test_fail_copy(int64_t nth_copy) { g_fail_copy.store(nth_copy > 0 ? nth_copy : 0); }

extern "C" int lema_stream_layers(lema_pool* pool, const lema_layer* layers, int32_t n_layers,
                                  int32_t residency, int32_t micro_step,
                                  const lema_adamw_hparams* hp, int64_t step, void* cuda_stream) {
    clear_error();
    if (!hp) return set_error(LEMA_ERR_ARG, "hparams is NULL");
    const int32_t K = hp->accum_steps;
    StepScalars s;
    LEMA_TRY(make_scalars(step, hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay, K, &s));
    if (micro_step < 1 || micro_step > K)
        return set_error(LEMA_ERR_ARG, "micro_step must lie in [1, accum_steps=%d] (got %d)", K,
                         micro_step);
    if (n_layers < 0) return set_error(LEMA_ERR_ARG, "n_layers must be >= 0");
    if (n_layers == 0) return LEMA_OK;
    if (!layers) return set_error(LEMA_ERR_ARG, "layers is NULL");
    for (int32_t L = 0; L < n_layers; ++L) {
        if (layers[L].count < 0) return set_error(LEMA_ERR_ARG, "unit %d: count must be >= 0", L);
        if (layers[L].count > 0 && (!layers[L].tensors || !layers[L].grads))
            return set_error(LEMA_ERR_ARG, "unit %d: NULL tensors or grads array", L);
    }
    const bool final_step = micro_step == K;
    cudaStream_t caller = static_cast<cudaStream_t>(cuda_stream);

    if (residency == LEMA_RESIDENT) {
        // Micro-step 1 starts the accumulator from +0.0 without reading it; the last
        // micro-step's grad is folded into an in-place step, which then resets acc.
        std::vector<lema_grad> g;
        std::vector<lema_tensor> t;
        for (int32_t L = 0; L < n_layers; ++L)
            for (int32_t j = 0; j < layers[L].count; ++j) {
                lema_tensor x = layers[L].tensors[j];
                x.flags = 0;
                x.grad_bf16 = final_step ? layers[L].grads[j] : nullptr;
                if (final_step && micro_step == 1) x.acc = nullptr;
                g.push_back(lema_grad{x.acc, layers[L].grads[j], x.n,
                                      micro_step == 1 ? int32_t(LEMA_GRAD_FIRST) : 0, 0});
                t.push_back(x);
            }
        if (!final_step) return lema_accum_grad(g.data(), int32_t(g.size()), cuda_stream);
        return lema_adamw_step(t.data(), int32_t(t.size()), step, hp->lr, hp->beta1, hp->beta2,
                               hp->eps, hp->weight_decay, K, cuda_stream);
    }
    if (residency != LEMA_STREAMED) return set_error(LEMA_ERR_ARG, "unknown residency %d", residency);
    if (!pool) return set_error(LEMA_ERR_ARG, "pool is NULL");
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
    if (device != pool->device)
        return set_error(LEMA_ERR_STATE, "pool lives on device %d, current device is %d",
                         pool->device, device);
    std::lock_guard<std::mutex> lock(pool->mu);
    return lema::stream_units_locked(pool, layers, n_layers, micro_step, K, s, caller, nullptr);
}

int lema::stream_units_locked(lema_pool* pool, const lema_layer* layers, int32_t n_layers,
                              int32_t micro_step, int32_t K, const StepScalars& s,
                              cudaStream_t caller, UnitHooks* hooks) {
    const bool final_step = micro_step == K;
    // Validate every unit before anything is enqueued.
    std::vector<std::vector<char>> grad_on_host(static_cast<size_t>(n_layers));
    std::vector<char> acc_dev(static_cast<size_t>(n_layers), 0);
    for (int32_t L = 0; L < n_layers; ++L) {
        bool on_device = false;
        LEMA_TRY(check_streamed_unit(layers[L], L, micro_step, final_step, pool->slot_params,
                                     grad_on_host[size_t(L)], pool->kinds, &on_device));
        acc_dev[size_t(L)] = on_device;
    }
    LEMA_TRY(bound_writers(pool));

    LEMA_TRY(begin_call(pool, n_layers, caller));

    const bool acc_in = micro_step >= 2;
    const auto H2D = cudaMemcpyHostToDevice;
    const auto D2H = cudaMemcpyDeviceToHost;
    std::vector<int64_t> off;
    std::vector<AccDesc> ad;
    std::vector<StepDesc> sd;
    std::vector<size_t> waits;
    int32_t slot_units = 0;   // units of this call that went through a slot so far
    for (int32_t L = 0; L < n_layers; ++L) {
        const lema_layer& ly = layers[L];
        // Accumulators in device memory stay there: read and written in place by the
        // kernels, never copied (only the host-resident ones cross the link).
        const bool dev_acc = acc_dev[size_t(L)] != 0;
        const bool acc_h2d = acc_in && !dev_acc;
        if (!final_step && dev_acc && !hooks &&
            std::none_of(grad_on_host[size_t(L)].begin(), grad_on_host[size_t(L)].end(),
                         [](char c) { return c != 0; })) {
            // Nothing of this micro-step crosses the link: the accumulate runs in place
            // on the compute stream without a slot, so a later call's loads into the
            // slots need not wait for it (its states stream in meanwhile).
            int tr = -1;
            LEMA_TRY(trace_open(pool, pool->cmp, LEMA_STAGE_COMPUTE, L, &tr));
            ad.clear();
            for (int32_t j = 0; j < ly.count; ++j) {
                const lema_tensor& t = ly.tensors[j];
                if (t.n == 0) continue;
                AccDesc a;
                a.acc_in = acc_in ? t.acc : nullptr;
                a.acc_out = t.acc;
                a.grad = ly.grads[j];
                a.n = t.n;
                ad.push_back(a);
            }
            if (!pool->copies_only) LEMA_TRY(run_accum(ad.data(), int32_t(ad.size()), pool->cmp));
            LEMA_TRY(trace_close(pool, pool->cmp, tr));
            continue;
        }
        Slot& sl = pool->slots[size_t(pool->next_slot % pool->n_slots)];
        pool->next_slot++;
        const bool first_unit = slot_units++ == 0;
        off.assign(size_t(ly.count), 0);
        for (int32_t j = 1; j < ly.count; ++j)
            off[size_t(j)] = off[size_t(j - 1)] + round_up(ly.tensors[j - 1].n, kTensorAlign);
        // A packed unit moves each field in one copy per slice spanning its non-empty
        // tensors (from the first one's pointer); otherwise one copy per tensor.
        const bool packed = (ly.flags & LEMA_UNIT_PACKED) != 0;
        int32_t first = -1, last = -1;
        for (int32_t j = 0; j < ly.count; ++j)
            if (ly.tensors[j].n > 0) {
                if (first < 0) first = j;
                last = j;
            }
        const int64_t base = first < 0 ? 0 : off[size_t(first)];
        const int64_t n_span = first < 0 ? 0 : off[size_t(last)] + ly.tensors[last].n - base;
        int64_t bound[kMaxSlices + 1];
        const int S = unit_slices(pool, packed, first_unit, n_span, bound);
        // The part of tensor j in slice q, as [lo, hi) within the tensor (all of it
        // when the unit is not sliced).
        auto part = [&](int32_t j, int q, int64_t* lo, int64_t* hi) {
            const int64_t n = ly.tensors[j].n, o = off[size_t(j)] - base;
            if (S == 1) { *lo = 0; *hi = n; return; }
            *lo = std::max<int64_t>(0, bound[q] - o);
            *hi = std::min<int64_t>(n, bound[q + 1] - o);
        };
        // the fields' copies of slice q: (slot offset, host element offset, count)
        auto field_copy = [&](int32_t j, int q, int64_t* o, int64_t* h, int64_t* n) {
            if (!packed) { *o = off[size_t(j)]; *h = 0; *n = ly.tensors[j].n; return; }
            if (j != first) { *n = 0; return; }
            *o = base + bound[q];
            *h = bound[q];
            *n = bound[q + 1] - bound[q];
        };

        // -- host -> device: the unit's inputs into the slot's input half (once a
        // lower tier, if any, has put them into the host buffers), slice by slice.
        if (hooks) LEMA_TRY(hooks->before_unit(L));
        LEMA_TRY(wait_on(pool->h2d, sl.step_done));
        waits.clear();
        for (int32_t j = 0; j < ly.count; ++j) {
            const lema_tensor& t = ly.tensors[j];
            const void* reads[] = {acc_h2d ? t.acc : nullptr, final_step ? t.master : nullptr,
                                   final_step ? t.m : nullptr, final_step ? t.v : nullptr};
            for (const void* p : reads) note_writer(pool, p, waits);
        }
        LEMA_TRY(wait_for_writers(pool, waits));
        for (int q = 0; q < S; ++q) {
            int tr = -1;
            LEMA_TRY(trace_open(pool, pool->h2d, LEMA_STAGE_H2D, L, &tr));
            for (int32_t j = 0; j < ly.count; ++j) {
                const lema_tensor& t = ly.tensors[j];
                int64_t lo = 0, hi = 0;
                part(j, q, &lo, &hi);
                if (grad_on_host[size_t(L)][size_t(j)] && hi > lo)
                    LEMA_TRY(copy_async(sl.grad + off[size_t(j)] + lo, ly.grads[j] + lo,
                                        2 * (hi - lo), H2D, pool->h2d));
                int64_t o = 0, h = 0, n = 0;
                field_copy(j, q, &o, &h, &n);
                if (n == 0) continue;
                if (acc_h2d) LEMA_TRY(copy_async(sl.acc + o, t.acc + h, 4 * n, H2D, pool->h2d));
                if (final_step) {
                    LEMA_TRY(copy_async(sl.master + o, t.master + h, 4 * n, H2D, pool->h2d));
                    LEMA_TRY(copy_async(sl.m + o, t.m + h, 4 * n, H2D, pool->h2d));
                    LEMA_TRY(copy_async(sl.v + o, t.v + h, 4 * n, H2D, pool->h2d));
                    LEMA_TRY(copy_async(sl.orig + o, t.orig_bf16 + h, 2 * n, H2D, pool->h2d));
                }
            }
            LEMA_TRY(trace_close(pool, pool->h2d, tr));
            LEMA_TRY(record(sl.in_ready[q], pool->h2d));
        }

        // -- compute, from the input half into the output half, slice by slice:
        // accumulate-only micro-steps add the grad into a new partial sum; the last
        // micro-step folds its grad into the out-of-place AdamW step (acc not written).
        LEMA_TRY(wait_on(pool->cmp, sl.out_drained));
        for (int q = 0; q < S; ++q) {
            LEMA_TRY(wait_on(pool->cmp, sl.in_ready[q]));
            int tr = -1;
            LEMA_TRY(trace_open(pool, pool->cmp, LEMA_STAGE_COMPUTE, L, &tr));
            ad.clear();
            sd.clear();
            for (int32_t j = 0; j < ly.count; ++j) {
                int64_t lo = 0, hi = 0;
                part(j, q, &lo, &hi);
                if (S > 1 && hi <= lo) continue;
                const int64_t o = off[size_t(j)] + lo;
                const uint16_t* g = grad_on_host[size_t(L)][size_t(j)] ? sl.grad + o
                                                                        : ly.grads[j] + lo;
                float* acc = !acc_in ? nullptr : dev_acc ? ly.tensors[j].acc + lo : sl.acc + o;
                if (!final_step) {
                    AccDesc a;
                    a.acc_in = acc;
                    a.acc_out = dev_acc ? ly.tensors[j].acc + lo : sl.delta + o;
                    a.grad = g;
                    a.n = hi - lo;
                    ad.push_back(a);
                } else {
                    StepDesc x;
                    x.master_in = sl.master + o;
                    x.m_in = sl.m + o;
                    x.v_in = sl.v + o;
                    x.acc = acc;
                    x.orig = sl.orig + o;
                    x.master_out = sl.master_o + o;
                    x.m_out = sl.m_o + o;
                    x.v_out = sl.v_o + o;
                    x.delta = sl.delta + o;
                    x.w = sl.w + o;
                    x.grad = g;
                    x.n = hi - lo;
                    x.flags = 0;
                    sd.push_back(x);
                }
            }
            if (!pool->copies_only) {
                if (!final_step) LEMA_TRY(run_accum(ad.data(), int32_t(ad.size()), pool->cmp));
                else LEMA_TRY(run_step(sd.data(), int32_t(sd.size()), s, pool->cmp));
            }
            LEMA_TRY(trace_close(pool, pool->cmp, tr));
            LEMA_TRY(record(sl.done[q], pool->cmp));
        }
        LEMA_TRY(record(sl.step_done, pool->cmp));

        // -- device -> host: results out of the slot's output half, slice by slice.
        // Every tensor's own host buffers name this unit as their writer (a packed
        // unit moves them in the first tensor's span copies), so a later call that
        // groups the tensors differently still waits for these copies.
        for (int32_t j = 0; j < ly.count; ++j) {
            const lema_tensor& t = ly.tensors[j];
            if (t.n == 0) continue;
            if (!final_step) {
                if (!dev_acc) pool->last_writer[t.acc] = size_t(L);
            } else {
                pool->last_writer[t.master_out ? t.master_out : t.master] = size_t(L);
                pool->last_writer[t.m_out ? t.m_out : t.m] = size_t(L);
                pool->last_writer[t.v_out ? t.v_out : t.v] = size_t(L);
            }
        }
        for (int q = 0; q < S; ++q) {
            LEMA_TRY(wait_on(pool->d2h, sl.done[q]));
            int tr = -1;
            LEMA_TRY(trace_open(pool, pool->d2h, LEMA_STAGE_D2H, L, &tr));
            for (int32_t j = 0; j < ly.count; ++j) {
                const lema_tensor& t = ly.tensors[j];
                int64_t o = 0, h = 0, n = 0;
                field_copy(j, q, &o, &h, &n);
                if (n == 0) continue;
                float* mo = t.master_out ? t.master_out : t.master;
                float* m_o = t.m_out ? t.m_out : t.m;
                float* v_o = t.v_out ? t.v_out : t.v;
                if (!final_step) {
                    if (!dev_acc)
                        LEMA_TRY(copy_async(t.acc + h, sl.delta + o, 4 * n, D2H, pool->d2h));
                } else {
                    LEMA_TRY(copy_async(mo + h, sl.master_o + o, 4 * n, D2H, pool->d2h));
                    LEMA_TRY(copy_async(m_o + h, sl.m_o + o, 4 * n, D2H, pool->d2h));
                    LEMA_TRY(copy_async(v_o + h, sl.v_o + o, 4 * n, D2H, pool->d2h));
                    LEMA_TRY(copy_async(t.delta + h, sl.delta + o, 4 * n, D2H, pool->d2h));
                    LEMA_TRY(copy_async(t.w_bf16 + h, sl.w + o, 2 * n, D2H, pool->d2h));
                }
            }
            LEMA_TRY(trace_close(pool, pool->d2h, tr));
        }
        LEMA_TRY(record(sl.out_drained, pool->d2h));
        LEMA_TRY(record(pool->unit_done[size_t(L)], pool->d2h));
        if (hooks) LEMA_TRY(hooks->after_unit(L, pool->d2h));
    }
    return end_call(pool);
}

int lema::pool_device(const lema_pool* pool) { return pool->device; }

namespace {

int bound_writers(lema_pool* pool) {
    constexpr size_t kMaxWriters = size_t(1) << 20;
    if (pool->last_writer.size() < kMaxWriters) return LEMA_OK;
    const auto deadline = std::chrono::steady_clock::now() + std::chrono::seconds(600);
    for (;;) {
        const cudaError_t e = cudaStreamQuery(pool->d2h);
        if (e == cudaSuccess) break;
        if (e != cudaErrorNotReady) return cuda_error(e, "pool device-to-host stream");
        if (std::chrono::steady_clock::now() >= deadline)
            return set_error(LEMA_ERR_TIMEOUT, "pool copies still pending while trimming its maps");
        std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
    pool->last_writer.clear();
    return LEMA_OK;
}

// The start of a streamed call: an event per unit index, and the pool's three
// streams ordered after the work the caller has enqueued so far.
int begin_call(lema_pool* pool, int32_t n_units, cudaStream_t caller) {
    while (pool->unit_done.size() < size_t(n_units)) {
        cudaEvent_t ev;
        LEMA_TRY(new_event(&ev));
        pool->unit_done.push_back(ev);
    }
    LEMA_TRY(record(pool->entry, caller));
    LEMA_TRY(wait_on(pool->h2d, pool->entry));
    LEMA_TRY(wait_on(pool->cmp, pool->entry));
    return wait_on(pool->d2h, pool->entry);
}

// Collect the unit (of an earlier call, or this one) whose device-to-host copies last
// wrote host buffer p.
void note_writer(lema_pool* pool, const void* p, std::vector<size_t>& waits) {
    if (!p) return;
    auto it = pool->last_writer.find(p);
    if (it != pool->last_writer.end()) waits.push_back(it->second);
}

// Make the host-to-device stream wait for those units' copies (each once).
int wait_for_writers(lema_pool* pool, std::vector<size_t>& waits) {
    std::sort(waits.begin(), waits.end());
    waits.erase(std::unique(waits.begin(), waits.end()), waits.end());
    for (size_t u : waits) LEMA_TRY(wait_on(pool->h2d, pool->unit_done[u]));
    return LEMA_OK;
}

// The end of a streamed call: the tail events lema_pool_sync and
// lema_pool_wait_stream wait on.
int end_call(lema_pool* pool) {
    LEMA_TRY(record(pool->tail[0], pool->h2d));
    LEMA_TRY(record(pool->tail[1], pool->cmp));
    LEMA_TRY(record(pool->tail[2], pool->d2h));
    pool->calls++;
    return LEMA_OK;
}

}  // namespace
std::mutex& lema::pool_mutex(lema_pool* pool) { return pool->mu; }

extern "C" int lema_pool_trace(lema_pool* pool, int32_t max_events) {
    clear_error();
    if (!pool) return set_error(LEMA_ERR_ARG, "pool is NULL");
    if (max_events < 0) return set_error(LEMA_ERR_ARG, "max_events must be >= 0");
    std::lock_guard<std::mutex> lock(pool->mu);
    LEMA_TRY(lema_pool_sync(pool, 600000));
    clear_trace(pool);
    pool->trace_cap = max_events;
    pool->calls = 0;
    return LEMA_OK;
}

extern "C" int lema_pool_trace_read(lema_pool* pool, lema_trace_event* out, int32_t max,
                                    int32_t* n_out) {
    clear_error();
    if (!pool || !n_out || (max > 0 && !out)) return set_error(LEMA_ERR_ARG, "NULL argument");
    LEMA_TRY(lema_pool_sync(pool, 600000));
    std::lock_guard<std::mutex> lock(pool->mu);
    const int32_t n = std::min<int32_t>(max, int32_t(pool->trace.size()));
    *n_out = int32_t(pool->trace.size());
    if (pool->trace.empty()) return LEMA_OK;
    // Times relative to the earliest stage start.
    cudaEvent_t ref = pool->trace[0].start;
    for (auto& r : pool->trace) {
        float d = 0.f;
        if (cudaEventElapsedTime(&d, ref, r.start) == cudaSuccess && d < 0.f) ref = r.start;
    }
    for (int32_t i = 0; i < n; ++i) {
        const auto& r = pool->trace[size_t(i)];
        float a = 0.f, b = 0.f;
        cudaError_t e = cudaEventElapsedTime(&a, ref, r.start);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&b, ref, r.end);
        if (e != cudaSuccess) return cuda_error(e, "cudaEventElapsedTime");
        out[i] = lema_trace_event{r.stage, r.unit, r.call, 0, double(a), double(b)};
    }
    return LEMA_OK;
}

// ======================================================= 8-bit streamed states ==
//
// The same pool, slots, streams, events and trace as lema_stream_layers, for units
// whose states are 8-bit (lema_tensor_q8).  A slot is re-carved for this layout
// (it fits in the 38 bytes per element of a slot; tensors of a unit sit at
// 1024-element offsets, so each tensor's block scales are a whole slice that
// starts on a 16-byte boundary):
//   input half : master fp32, m_q, r_q, acc_q (1 B), orig, grad (bf16), and the
//                m, r, acc block scales (fp32 per 256 elements)
//   output half: master' fp32, m_q', r_q', acc_q' (1 B), delta fp32, w bf16, and
//                the m', r', acc' block scales
// Accumulate-only micro-steps write acc' to the output half; the last micro-step
// folds its grad into the out-of-place 8-bit step.

namespace {

constexpr int64_t kQAlign = 4 * kQBlock;   // tensor offsets inside a unit, in elements

struct SlotQ8 {
    float* master;
    int8_t* m_q;
    uint8_t* r_q;
    int8_t* acc_q;
    uint16_t* orig;
    uint16_t* grad;
    float* m_s;
    float* r_s;
    float* acc_s;
    float* master_o;
    int8_t* m_q_o;
    uint8_t* r_q_o;
    int8_t* acc_q_o;
    float* delta;
    uint16_t* w;
    float* m_s_o;
    float* r_s_o;
    float* acc_s_o;
};

SlotQ8 carve_q8(const Slot& s, int64_t P) {
    unsigned char* b = reinterpret_cast<unsigned char*>(s.master);   // the slot's base
    const int64_t nb = (P + kQBlock - 1) / kQBlock;
    auto take = [&](int64_t bytes) {
        unsigned char* p = b;
        b += (bytes + 255) / 256 * 256;
        return p;
    };
    SlotQ8 q;
    q.master = reinterpret_cast<float*>(take(4 * P));
    q.m_q = reinterpret_cast<int8_t*>(take(P));
    q.r_q = reinterpret_cast<uint8_t*>(take(P));
    q.acc_q = reinterpret_cast<int8_t*>(take(P));
    q.orig = reinterpret_cast<uint16_t*>(take(2 * P));
    q.grad = reinterpret_cast<uint16_t*>(take(2 * P));
    q.m_s = reinterpret_cast<float*>(take(4 * nb));
    q.r_s = reinterpret_cast<float*>(take(4 * nb));
    q.acc_s = reinterpret_cast<float*>(take(4 * nb));
    q.master_o = reinterpret_cast<float*>(take(4 * P));
    q.m_q_o = reinterpret_cast<int8_t*>(take(P));
    q.r_q_o = reinterpret_cast<uint8_t*>(take(P));
    q.acc_q_o = reinterpret_cast<int8_t*>(take(P));
    q.delta = reinterpret_cast<float*>(take(4 * P));
    q.w = reinterpret_cast<uint16_t*>(take(2 * P));
    q.m_s_o = reinterpret_cast<float*>(take(4 * nb));
    q.r_s_o = reinterpret_cast<float*>(take(4 * nb));
    q.acc_s_o = reinterpret_cast<float*>(take(4 * nb));
    return q;
}

// Bytes carve_q8 uses for a slot of P elements (the pool sizes each slot for the
// larger of this and the fp32 layout's 38 P).
int64_t carved_q8_bytes(int64_t P) {
    const int64_t nb = (P + kQBlock - 1) / kQBlock;
    auto r = [](int64_t x) { return (x + 255) / 256 * 256; };
    return 2 * r(4 * P) + 6 * r(P) + 2 * r(2 * P) + r(4 * P) + r(2 * P) + 6 * r(4 * nb);
}

int check_streamed_unit_q8(const lema_layer_q8& ly, int32_t L, bool final_step,
                           int64_t slot_params, std::vector<char>& grad_on_host,
                           std::unordered_map<const void*, int>& kinds, bool* acc_on_device) {
    int64_t need = 0;
    int acc_kind = 0;
    for (int32_t j = 0; j < ly.count; ++j) {
        const lema_tensor_q8& t = ly.tensors[j];
        if (t.n < 0) return set_error(LEMA_ERR_ARG, "unit %d tensor %d: n must be >= 0", L, j);
        need += round_up(t.n, kQAlign);
        grad_on_host.push_back(0);
        if (t.n == 0) continue;
        const int outs = (t.master_out != nullptr) + (t.m_q_out != nullptr) +
                         (t.m_scale_out != nullptr) + (t.r_q_out != nullptr) +
                         (t.r_scale_out != nullptr);
        if (outs != 0 && outs != 5)
            return set_error(LEMA_ERR_ARG,
                             "unit %d tensor %d: the five *_out fields must be all NULL or all set",
                             L, j);
        const void* acc[] = {t.acc_q, t.acc_scale};
        LEMA_TRY(check_acc_kind(acc, 2, L, j, kinds, &acc_kind));
        std::vector<const void*> host;
        if (final_step) {
            host.insert(host.end(), {t.master, t.m_q, t.m_scale, t.r_q, t.r_scale, t.orig_bf16,
                                     t.delta, t.w_bf16});
            if (outs)
                host.insert(host.end(),
                            {t.master_out, t.m_q_out, t.m_scale_out, t.r_q_out, t.r_scale_out});
        }
        for (const void* p : host) {
            if (!p) return set_error(LEMA_ERR_ARG, "unit %d tensor %d: NULL host buffer", L, j);
            if (!aligned16(p))
                return set_error(LEMA_ERR_ALIGN, "unit %d tensor %d: host buffer not 16-byte aligned",
                                 L, j);
            if (cached_kind(kinds, p) != 1)
                return set_error(LEMA_ERR_ARG,
                                 "unit %d tensor %d: state buffers must be pinned host memory", L, j);
        }
        const uint16_t* g = ly.grads[j];
        if (!g) return set_error(LEMA_ERR_ARG, "unit %d tensor %d: NULL grad", L, j);
        if (!aligned16(g))
            return set_error(LEMA_ERR_ALIGN, "unit %d tensor %d: grad not 16-byte aligned", L, j);
        const int kind = cached_kind(kinds, g);
        if (kind == 0)
            return set_error(LEMA_ERR_ARG,
                             "unit %d tensor %d: grad must be memory of the pool's GPU or pinned "
                             "host memory", L, j);
        grad_on_host.back() = (kind == 1);
    }
    *acc_on_device = acc_kind == 2;
    if (need > slot_params)
        return set_error(LEMA_ERR_ARG, "unit %d needs %lld slot elements, a slot holds %lld", L,
                         (long long)need, (long long)slot_params);
    if (ly.flags & ~int32_t(LEMA_UNIT_PACKED))
        return set_error(LEMA_ERR_ARG, "unit %d: unknown flags", L);
    if (ly.flags & LEMA_UNIT_PACKED) {
        int32_t first = -1;
        int64_t o = 0, o_first = 0;
        for (int32_t j = 0; j < ly.count; ++j) {
            const lema_tensor_q8& t = ly.tensors[j];
            const int64_t oj = o;
            o += round_up(t.n, kQAlign);
            if (t.n == 0) continue;
            if (first < 0) {
                first = j;
                o_first = oj;
            }
            const lema_tensor_q8& t0 = ly.tensors[first];
            const int64_t de = oj - o_first, db = de / kQBlock;
            auto at = [](const void* base, const void* p, int64_t bytes) {
                return reinterpret_cast<uintptr_t>(p) == reinterpret_cast<uintptr_t>(base) + uintptr_t(bytes);
            };
            bool ok = *acc_on_device ||
                      (at(t0.acc_q, t.acc_q, de) && at(t0.acc_scale, t.acc_scale, 4 * db));
            if (final_step) {
                ok = ok && at(t0.master, t.master, 4 * de) && at(t0.m_q, t.m_q, de) &&
                     at(t0.m_scale, t.m_scale, 4 * db) && at(t0.r_q, t.r_q, de) &&
                     at(t0.r_scale, t.r_scale, 4 * db) && at(t0.orig_bf16, t.orig_bf16, 2 * de) &&
                     at(t0.delta, t.delta, 4 * de) && at(t0.w_bf16, t.w_bf16, 2 * de);
                if (t0.master_out)
                    ok = ok && at(t0.master_out, t.master_out, 4 * de) &&
                         at(t0.m_q_out, t.m_q_out, de) && at(t0.m_scale_out, t.m_scale_out, 4 * db) &&
                         at(t0.r_q_out, t.r_q_out, de) && at(t0.r_scale_out, t.r_scale_out, 4 * db);
            }
            if (!ok)
                return set_error(LEMA_ERR_ARG,
                                 "unit %d is flagged packed but tensor %d is not at its slot offset",
                                 L, j);
        }
    }
    return LEMA_OK;
}

}  // namespace

extern "C" int lema_stream_layers_q8(lema_pool* pool, const lema_layer_q8* layers,
                                     int32_t n_layers, int32_t micro_step,
                                     const lema_adamw_hparams* hp, int64_t step,
                                     void* cuda_stream) {
    clear_error();
    if (!hp) return set_error(LEMA_ERR_ARG, "hparams is NULL");
    const int32_t K = hp->accum_steps;
    StepScalars s;
    LEMA_TRY(make_scalars(step, hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay, K, &s));
    if (micro_step < 1 || micro_step > K)
        return set_error(LEMA_ERR_ARG, "micro_step must lie in [1, accum_steps=%d] (got %d)", K,
                         micro_step);
    if (n_layers < 0) return set_error(LEMA_ERR_ARG, "n_layers must be >= 0");
    if (n_layers == 0) return LEMA_OK;
    if (!layers) return set_error(LEMA_ERR_ARG, "layers is NULL");
    if (!pool) return set_error(LEMA_ERR_ARG, "pool is NULL");
    for (int32_t L = 0; L < n_layers; ++L) {
        if (layers[L].count < 0) return set_error(LEMA_ERR_ARG, "unit %d: count must be >= 0", L);
        if (layers[L].count > 0 && (!layers[L].tensors || !layers[L].grads))
            return set_error(LEMA_ERR_ARG, "unit %d: NULL tensors or grads array", L);
    }
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
    if (device != pool->device)
        return set_error(LEMA_ERR_STATE, "pool lives on device %d, current device is %d",
                         pool->device, device);
    cudaStream_t caller = static_cast<cudaStream_t>(cuda_stream);
    std::lock_guard<std::mutex> lock(pool->mu);
    return lema::stream_units_q8_locked(pool, layers, n_layers, micro_step, K, s, caller, nullptr);
}

int lema::stream_units_q8_locked(lema_pool* pool, const lema_layer_q8* layers, int32_t n_layers,
                                 int32_t micro_step, int32_t K, const StepScalars& s,
                                 cudaStream_t caller, UnitHooks* hooks) {
    if (carved_q8_bytes(pool->slot_params) > pool->slot_bytes)
        return set_error(LEMA_ERR_STATE, "slot too small for the 8-bit layout");
    // A give-up in an earlier call that nobody has synced on yet: report it first.
    LEMA_TRY(gave_up_take(pool->gave_up, "8-bit streamed call (an earlier call of this pool; "
                                         "nothing was enqueued now)"));
    const bool final_step = micro_step == K;
    const bool acc_in = micro_step >= 2;
    std::vector<std::vector<char>> grad_on_host(static_cast<size_t>(n_layers));
    std::vector<char> acc_dev(static_cast<size_t>(n_layers), 0);
    for (int32_t L = 0; L < n_layers; ++L) {
        bool on_device = false;
        LEMA_TRY(check_streamed_unit_q8(layers[L], L, final_step, pool->slot_params,
                                        grad_on_host[size_t(L)], pool->kinds, &on_device));
        acc_dev[size_t(L)] = on_device;
    }
    LEMA_TRY(bound_writers(pool));
    LEMA_TRY(begin_call(pool, n_layers, caller));

    std::vector<int64_t> off;
    std::vector<AccDescQ8> ad;
    std::vector<StepDescQ8> sd;
    std::vector<size_t> waits;
    int32_t slot_units = 0;
    const auto H2D = cudaMemcpyHostToDevice;
    const auto D2H = cudaMemcpyDeviceToHost;
    auto blocks = [](int64_t n) { return (n + kQBlock - 1) / kQBlock; };
    for (int32_t L = 0; L < n_layers; ++L) {
        const lema_layer_q8& ly = layers[L];
        const bool dev_acc = acc_dev[size_t(L)] != 0;   // as in lema_stream_layers
        const bool acc_h2d = acc_in && !dev_acc;
        if (!final_step && dev_acc && !hooks &&
            std::none_of(grad_on_host[size_t(L)].begin(), grad_on_host[size_t(L)].end(),
                         [](char c) { return c != 0; })) {
            // an accumulate that moves nothing: in place, no slot (lema_stream_layers)
            int tr = -1;
            LEMA_TRY(trace_open(pool, pool->cmp, LEMA_STAGE_COMPUTE, L, &tr));
            ad.clear();
            for (int32_t j = 0; j < ly.count; ++j) {
                const lema_tensor_q8& t = ly.tensors[j];
                if (t.n == 0) continue;
                AccDescQ8 a;
                a.acc_q_in = acc_in ? t.acc_q : nullptr;
                a.acc_scale_in = acc_in ? t.acc_scale : nullptr;
                a.acc_q_out = t.acc_q;
                a.acc_scale_out = t.acc_scale;
                a.grad = ly.grads[j];
                a.n = t.n;
                ad.push_back(a);
            }
            if (!pool->copies_only)
                LEMA_TRY(run_accum_q8(ad.data(), int32_t(ad.size()), pool->cmp));
            LEMA_TRY(trace_close(pool, pool->cmp, tr));
            continue;
        }
        Slot& sl0 = pool->slots[size_t(pool->next_slot % pool->n_slots)];
        pool->next_slot++;
        const bool first_unit = slot_units++ == 0;
        const SlotQ8 sl = carve_q8(sl0, pool->slot_params);
        off.assign(size_t(ly.count), 0);
        for (int32_t j = 1; j < ly.count; ++j)
            off[size_t(j)] = off[size_t(j - 1)] + round_up(ly.tensors[j - 1].n, kQAlign);
        const bool packed = (ly.flags & LEMA_UNIT_PACKED) != 0;
        int32_t first = -1, last = -1;
        for (int32_t j = 0; j < ly.count; ++j)
            if (ly.tensors[j].n > 0) {
                if (first < 0) first = j;
                last = j;
            }
        // The packed span starts at the first non-empty tensor (a multiple of 1024
        // elements), so every slice boundary (whole chunks) is a whole number of
        // blocks and each slice's scales start on a 16-byte boundary.
        const int64_t base = first < 0 ? 0 : off[size_t(first)];
        const int64_t n_span = first < 0 ? 0 : off[size_t(last)] + ly.tensors[last].n - base;
        int64_t bound[kMaxSlices + 1];
        const int S = unit_slices(pool, packed, first_unit, n_span, bound);
        auto part = [&](int32_t j, int q, int64_t* lo, int64_t* hi) {
            const int64_t n = ly.tensors[j].n, o = off[size_t(j)] - base;
            if (S == 1) { *lo = 0; *hi = n; return; }
            *lo = std::max<int64_t>(0, bound[q] - o);
            *hi = std::min<int64_t>(n, bound[q + 1] - o);
        };
        // slice q's copies of tensor j: slot offset o, host element offset h, n
        // elements and nb scales (a packed unit: one span from its first tensor)
        auto field_copy = [&](int32_t j, int q, int64_t* o, int64_t* h, int64_t* n,
                              int64_t* nb) {
            if (!packed) {
                *o = off[size_t(j)];
                *h = 0;
                *n = ly.tensors[j].n;
                *nb = blocks(*n);
                return;
            }
            if (j != first) { *n = *nb = 0; return; }
            *o = base + bound[q];
            *h = bound[q];
            *n = bound[q + 1] - bound[q];
            *nb = blocks(bound[q + 1]) - bound[q] / kQBlock;
        };

        // -- host -> device (once a lower tier, if any, has filled the host buffers)
        if (hooks) LEMA_TRY(hooks->before_unit(L));
        LEMA_TRY(wait_on(pool->h2d, sl0.step_done));
        waits.clear();
        for (int32_t j = 0; j < ly.count; ++j) {
            const lema_tensor_q8& t = ly.tensors[j];
            const void* reads[] = {acc_h2d ? t.acc_q : nullptr, final_step ? t.master : nullptr,
                                   final_step ? t.m_q : nullptr, final_step ? t.r_q : nullptr};
            for (const void* p : reads) note_writer(pool, p, waits);
        }
        LEMA_TRY(wait_for_writers(pool, waits));
        for (int q = 0; q < S; ++q) {
            int tr = -1;
            LEMA_TRY(trace_open(pool, pool->h2d, LEMA_STAGE_H2D, L, &tr));
            for (int32_t j = 0; j < ly.count; ++j) {
                const lema_tensor_q8& t = ly.tensors[j];
                int64_t lo = 0, hi = 0;
                part(j, q, &lo, &hi);
                if (grad_on_host[size_t(L)][size_t(j)] && hi > lo)
                    LEMA_TRY(copy_async(sl.grad + off[size_t(j)] + lo, ly.grads[j] + lo,
                                        2 * (hi - lo), H2D, pool->h2d));
                int64_t o = 0, h = 0, n = 0, nb = 0;
                field_copy(j, q, &o, &h, &n, &nb);
                if (n == 0) continue;
                const int64_t b = o / kQBlock, hb = h / kQBlock;
                if (acc_h2d) {
                    LEMA_TRY(copy_async(sl.acc_q + o, t.acc_q + h, n, H2D, pool->h2d));
                    LEMA_TRY(copy_async(sl.acc_s + b, t.acc_scale + hb, 4 * nb, H2D, pool->h2d));
                }
                if (final_step) {
                    LEMA_TRY(copy_async(sl.master + o, t.master + h, 4 * n, H2D, pool->h2d));
                    LEMA_TRY(copy_async(sl.m_q + o, t.m_q + h, n, H2D, pool->h2d));
                    LEMA_TRY(copy_async(sl.m_s + b, t.m_scale + hb, 4 * nb, H2D, pool->h2d));
                    LEMA_TRY(copy_async(sl.r_q + o, t.r_q + h, n, H2D, pool->h2d));
                    LEMA_TRY(copy_async(sl.r_s + b, t.r_scale + hb, 4 * nb, H2D, pool->h2d));
                    LEMA_TRY(copy_async(sl.orig + o, t.orig_bf16 + h, 2 * n, H2D, pool->h2d));
                }
            }
            LEMA_TRY(trace_close(pool, pool->h2d, tr));
            LEMA_TRY(record(sl0.in_ready[q], pool->h2d));
        }

        // -- compute, slice by slice
        LEMA_TRY(wait_on(pool->cmp, sl0.out_drained));
        for (int q = 0; q < S; ++q) {
            LEMA_TRY(wait_on(pool->cmp, sl0.in_ready[q]));
            int tr = -1;
            LEMA_TRY(trace_open(pool, pool->cmp, LEMA_STAGE_COMPUTE, L, &tr));
            ad.clear();
            sd.clear();
            for (int32_t j = 0; j < ly.count; ++j) {
                int64_t lo = 0, hi = 0;
                part(j, q, &lo, &hi);
                if (S > 1 && hi <= lo) continue;
                const int64_t o = off[size_t(j)] + lo, b = o / kQBlock;
                const uint16_t* g = grad_on_host[size_t(L)][size_t(j)] ? sl.grad + o
                                                                        : ly.grads[j] + lo;
                // a device-resident accumulator: tensor j's own codes and scales
                // (lo is a whole number of blocks: slice bounds are whole chunks)
                const lema_tensor_q8& t = ly.tensors[j];
                int8_t* acc_q = !acc_in ? nullptr : dev_acc ? t.acc_q + lo : sl.acc_q + o;
                float* acc_s = !acc_in ? nullptr : dev_acc ? t.acc_scale + lo / kQBlock
                                                           : sl.acc_s + b;
                if (!final_step) {
                    AccDescQ8 a;
                    a.acc_q_in = acc_q;
                    a.acc_scale_in = acc_s;
                    a.acc_q_out = dev_acc ? t.acc_q + lo : sl.acc_q_o + o;
                    a.acc_scale_out = dev_acc ? t.acc_scale + lo / kQBlock : sl.acc_s_o + b;
                    a.grad = g;
                    a.n = hi - lo;
                    ad.push_back(a);
                } else {
                    StepDescQ8 x;
                    x.master_in = sl.master + o;
                    x.m_q_in = sl.m_q + o;
                    x.m_scale_in = sl.m_s + b;
                    x.r_q_in = sl.r_q + o;
                    x.r_scale_in = sl.r_s + b;
                    x.acc_q = acc_q;
                    x.acc_scale = acc_s;
                    x.grad = g;
                    x.orig = sl.orig + o;
                    x.master_out = sl.master_o + o;
                    x.m_q_out = sl.m_q_o + o;
                    x.m_scale_out = sl.m_s_o + b;
                    x.r_q_out = sl.r_q_o + o;
                    x.r_scale_out = sl.r_s_o + b;
                    x.delta = sl.delta + o;
                    x.w = sl.w + o;
                    x.n = hi - lo;
                    x.flags = 0;
                    sd.push_back(x);
                }
            }
            if (!pool->copies_only) {
                if (!final_step)
                    LEMA_TRY(run_accum_q8(ad.data(), int32_t(ad.size()), pool->cmp));
                else
                    LEMA_TRY(run_step_q8(sd.data(), int32_t(sd.size()), s, pool->cmp,
                                         pool->gave_up.dev));
            }
            LEMA_TRY(trace_close(pool, pool->cmp, tr));
            LEMA_TRY(record(sl0.done[q], pool->cmp));
        }
        LEMA_TRY(record(sl0.step_done, pool->cmp));

        // -- device -> host, slice by slice (every tensor's own buffers name this unit
        // as their writer, as in lema_stream_layers)
        for (int32_t j = 0; j < ly.count; ++j) {
            const lema_tensor_q8& t = ly.tensors[j];
            if (t.n == 0) continue;
            if (!final_step) {
                if (!dev_acc) pool->last_writer[t.acc_q] = size_t(L);
            } else {
                pool->last_writer[t.master_out ? t.master_out : t.master] = size_t(L);
                pool->last_writer[t.m_q_out ? t.m_q_out : t.m_q] = size_t(L);
                pool->last_writer[t.r_q_out ? t.r_q_out : t.r_q] = size_t(L);
            }
        }
        for (int q = 0; q < S; ++q) {
            LEMA_TRY(wait_on(pool->d2h, sl0.done[q]));
            int tr = -1;
            LEMA_TRY(trace_open(pool, pool->d2h, LEMA_STAGE_D2H, L, &tr));
            for (int32_t j = 0; j < ly.count; ++j) {
                const lema_tensor_q8& t = ly.tensors[j];
                int64_t o = 0, h = 0, n = 0, nb = 0;
                field_copy(j, q, &o, &h, &n, &nb);
                if (n == 0) continue;
                const int64_t b = o / kQBlock, hb = h / kQBlock;
                float* mo = t.master_out ? t.master_out : t.master;
                int8_t* mq = t.m_q_out ? t.m_q_out : t.m_q;
                float* ms = t.m_scale_out ? t.m_scale_out : t.m_scale;
                uint8_t* rq = t.r_q_out ? t.r_q_out : t.r_q;
                float* rs = t.r_scale_out ? t.r_scale_out : t.r_scale;
                if (!final_step) {
                    if (!dev_acc) {
                        LEMA_TRY(copy_async(t.acc_q + h, sl.acc_q_o + o, n, D2H, pool->d2h));
                        LEMA_TRY(copy_async(t.acc_scale + hb, sl.acc_s_o + b, 4 * nb, D2H,
                                            pool->d2h));
                    }
                } else {
                    LEMA_TRY(copy_async(mo + h, sl.master_o + o, 4 * n, D2H, pool->d2h));
                    LEMA_TRY(copy_async(mq + h, sl.m_q_o + o, n, D2H, pool->d2h));
                    LEMA_TRY(copy_async(ms + hb, sl.m_s_o + b, 4 * nb, D2H, pool->d2h));
                    LEMA_TRY(copy_async(rq + h, sl.r_q_o + o, n, D2H, pool->d2h));
                    LEMA_TRY(copy_async(rs + hb, sl.r_s_o + b, 4 * nb, D2H, pool->d2h));
                    LEMA_TRY(copy_async(t.delta + h, sl.delta + o, 4 * n, D2H, pool->d2h));
                    LEMA_TRY(copy_async(t.w_bf16 + h, sl.w + o, 2 * n, D2H, pool->d2h));
                }
            }
            LEMA_TRY(trace_close(pool, pool->d2h, tr));
        }
        LEMA_TRY(record(sl0.out_drained, pool->d2h));
        LEMA_TRY(record(pool->unit_done[size_t(L)], pool->d2h));
        if (hooks) LEMA_TRY(hooks->after_unit(L, pool->d2h));
    }
    return end_call(pool);
}
