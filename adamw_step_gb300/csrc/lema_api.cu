// lema_api.cu -- host side of lema_accum_grad / lema_adamw_step: argument checks,
// the per-call fp32 scalars, the cached device descriptor tables and the launches.
//
// Page "LEMA: Layer-wise Efficient Memory Abstraction", sections "Selective Full
// Fine-Tuning" (fp32 accumulation, per-layer AdamW, fp32 delta) and "Quick Start"
// (torch.optim.AdamW: bias correction and decoupled weight decay).
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <deque>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "lema_internal.h"
#include "lema_q8.h"

namespace lema {

// ------------------------------------------------------------------ errors ----

static thread_local char g_err[512] = "";

int set_error(int status, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return status;
}

void clear_error() { g_err[0] = '\0'; }

int cuda_error(cudaError_t e, const char* what) {
    if (e == cudaErrorMemoryAllocation)
        return set_error(LEMA_ERR_OOM, "%s: %s", what, cudaGetErrorString(e));
    return set_error(LEMA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ----------------------------------------------------------------- scalars ----

int make_scalars(int64_t step, double lr, double beta1, double beta2, double eps,
                 double weight_decay, int32_t accum_steps, StepScalars* s) {
    if (step < 1) return set_error(LEMA_ERR_ARG, "step must be >= 1 (got %lld)", (long long)step);
    if (accum_steps < 1)
        return set_error(LEMA_ERR_ARG, "accum_steps must be >= 1 (got %d)", accum_steps);
    if (!(beta1 >= 0.0 && beta1 < 1.0) || !(beta2 >= 0.0 && beta2 < 1.0))
        return set_error(LEMA_ERR_ARG, "betas must lie in [0, 1) (got %g, %g)", beta1, beta2);
    if (!(eps > 0.0)) return set_error(LEMA_ERR_ARG, "eps must be > 0 (got %g)", eps);
    if (!(lr >= 0.0)) return set_error(LEMA_ERR_ARG, "lr must be >= 0 (got %g)", lr);
    if (!(weight_decay >= 0.0))
        return set_error(LEMA_ERR_ARG, "weight_decay must be >= 0 (got %g)", weight_decay);
    if (!(lr * weight_decay < 1.0))
        return set_error(LEMA_ERR_ARG, "lr*weight_decay must be < 1 (got %g)", lr * weight_decay);

    // beta^t, one fp64 factor at a time.  Once both products are below 2^-60 every
    // further product stays below it and 1 - p rounds to exactly 1.0, so the loop
    // may stop there without changing any result.
    double p1 = 1.0, p2 = 1.0;
    for (int64_t i = 0; i < step; ++i) {
        p1 *= beta1;
        p2 *= beta2;
        if (p1 < 0x1p-60 && p2 < 0x1p-60) break;
    }
    const double bc1 = 1.0 - p1, bc2 = 1.0 - p2;
    s->decay = float(1.0 - lr * weight_decay);
    s->beta1 = float(beta1);
    s->omb1 = float(1.0 - beta1);
    s->beta2 = float(beta2);
    s->omb2 = float(1.0 - beta2);
    s->step_size = float(lr / bc1);
    s->bc2_sqrt = float(std::sqrt(bc2));
    s->eps = float(eps);
    s->accum = float(accum_steps);
    const bool pow2 = (accum_steps & (accum_steps - 1)) == 0;
    s->accum_pow2 = pow2 ? 1 : 0;
    s->inv_accum = pow2 ? 1.0f / float(accum_steps) : 0.0f;
    s->bc2_rcp = rcp_rn(s->bc2_sqrt);
    return LEMA_OK;
}

float rcp_rn(float c) {
    // 1/c in fp64 is within 2^-53 (relative) of the exact reciprocal, and no exact
    // reciprocal of a 24-bit significand lies that close to a point halfway between
    // two fp32 numbers, so rounding it to fp32 is already correct; the neighbours are
    // still compared, exactly (c * r needs 48 bits, so fp64 holds it and 1 - c * r
    // without error), so that the result does not rest on that argument.
    float r = float(1.0 / double(c));
    const float cand[2] = {std::nextafter(r, 0.0f), std::nextafter(r, HUGE_VALF)};
    for (float x : cand)
        if (std::fabs(1.0 - double(c) * double(x)) < std::fabs(1.0 - double(c) * double(r))) r = x;
    return r;
}

// ------------------------------------------------------ overlap validation ----

namespace {

struct Span {
    uintptr_t lo, hi;  // [lo, hi)
    bool written;
    int32_t tensor;
    const char* field;
};

void add_span(std::vector<Span>& v, const void* p, int64_t bytes, bool written, int32_t t,
              const char* f) {
    if (bytes <= 0 || p == nullptr) return;
    uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    v.push_back(Span{lo, lo + uintptr_t(bytes), written, t, f});
}

// Any two spans that overlap where at least one is written is an error.
int check_spans(std::vector<Span>& v) {
    std::sort(v.begin(), v.end(), [](const Span& a, const Span& b) { return a.lo < b.lo; });
    uintptr_t max_end_any = 0, max_end_written = 0;
    const Span* owner_any = nullptr;
    const Span* owner_written = nullptr;
    for (const Span& s : v) {
        const Span* hit = nullptr;
        if (s.written && s.lo < max_end_any) hit = owner_any;
        else if (!s.written && s.lo < max_end_written) hit = owner_written;
        if (hit)
            return set_error(LEMA_ERR_ARG,
                             "buffers overlap: tensor %d %s and tensor %d %s (an output may "
                             "alias only its own input, in place)",
                             hit->tensor, hit->field, s.tensor, s.field);
        if (s.hi > max_end_any) { max_end_any = s.hi; owner_any = &s; }
        if (s.written && s.hi > max_end_written) { max_end_written = s.hi; owner_written = &s; }
    }
    return LEMA_OK;
}

int validate_step(const StepDesc* d, int32_t count) {
    std::vector<Span> v;
    v.reserve(size_t(count) * 10);
    for (int32_t j = 0; j < count; ++j) {
        const int64_t n = d[j].n, b4 = n * 4, b2 = n * 2;
        auto pair = [&](const float* in, float* out, const char* f) {
            if (in == out) add_span(v, in, b4, true, j, f);
            else { add_span(v, in, b4, false, j, f); add_span(v, out, b4, true, j, f); }
        };
        pair(d[j].master_in, d[j].master_out, "master");
        pair(d[j].m_in, d[j].m_out, "m");
        pair(d[j].v_in, d[j].v_out, "v");
        add_span(v, d[j].acc, b4, (d[j].flags & kZeroAcc) != 0, j, "acc");
        add_span(v, d[j].grad, b2, false, j, "grad_bf16");
        add_span(v, d[j].orig, b2, false, j, "orig_bf16");
        add_span(v, d[j].delta, b4, true, j, "delta");
        add_span(v, d[j].w, b2, true, j, "w_bf16");
    }
    return check_spans(v);
}

int validate_accum(const AccDesc* d, int32_t count) {
    std::vector<Span> v;
    v.reserve(size_t(count) * 3);
    for (int32_t j = 0; j < count; ++j) {
        const int64_t n = d[j].n;
        if (d[j].acc_in == d[j].acc_out) {
            add_span(v, d[j].acc_out, n * 4, true, j, "acc");
        } else {
            add_span(v, d[j].acc_in, n * 4, false, j, "acc_in");
            add_span(v, d[j].acc_out, n * 4, true, j, "acc_out");
        }
        add_span(v, d[j].grad, n * 2, false, j, "grad_bf16");
    }
    return check_spans(v);
}

int64_t q8_blocks(int64_t n) { return (n + kQBlock - 1) / kQBlock; }

int validate_step_q8(const StepDescQ8* d, int32_t count) {
    std::vector<Span> v;
    v.reserve(size_t(count) * 16);
    for (int32_t j = 0; j < count; ++j) {
        const int64_t n = d[j].n, nb4 = q8_blocks(n) * 4;
        auto pair = [&](const void* in, const void* out, int64_t bytes, const char* f) {
            if (in == out) add_span(v, in, bytes, true, j, f);
            else { add_span(v, in, bytes, false, j, f); add_span(v, out, bytes, true, j, f); }
        };
        pair(d[j].master_in, d[j].master_out, n * 4, "master");
        pair(d[j].m_q_in, d[j].m_q_out, n, "m_q");
        pair(d[j].m_scale_in, d[j].m_scale_out, nb4, "m_scale");
        pair(d[j].r_q_in, d[j].r_q_out, n, "r_q");
        pair(d[j].r_scale_in, d[j].r_scale_out, nb4, "r_scale");
        const bool zero = (d[j].flags & kZeroAcc) != 0;
        add_span(v, d[j].acc_q, n, zero, j, "acc_q");
        add_span(v, d[j].acc_scale, nb4, zero, j, "acc_scale");
        add_span(v, d[j].grad, n * 2, false, j, "grad_bf16");
        add_span(v, d[j].orig, n * 2, false, j, "orig_bf16");
        add_span(v, d[j].delta, n * 4, true, j, "delta");
        add_span(v, d[j].w, n * 2, true, j, "w_bf16");
    }
    return check_spans(v);
}

int validate_merge(const MergeDesc* d, int32_t count) {
    std::vector<Span> v;
    v.reserve(size_t(count) * 3);
    for (int32_t j = 0; j < count; ++j) {
        const int64_t n = d[j].n;
        if (d[j].base == d[j].merged) {
            add_span(v, d[j].merged, n * 2, true, j, "merged (in place)");
        } else {
            add_span(v, d[j].base, n * 2, false, j, "base_bf16");
            add_span(v, d[j].merged, n * 2, true, j, "merged_bf16");
        }
        add_span(v, d[j].delta, n * 4, false, j, "delta");
    }
    return check_spans(v);
}

int validate_accum_q8(const AccDescQ8* d, int32_t count) {
    std::vector<Span> v;
    v.reserve(size_t(count) * 5);
    for (int32_t j = 0; j < count; ++j) {
        const int64_t n = d[j].n, nb4 = q8_blocks(n) * 4;
        if (d[j].acc_q_in == d[j].acc_q_out) {
            add_span(v, d[j].acc_q_out, n, true, j, "acc_q");
            add_span(v, d[j].acc_scale_out, nb4, true, j, "acc_scale");
        } else {
            add_span(v, d[j].acc_q_in, n, false, j, "acc_q_in");
            add_span(v, d[j].acc_scale_in, nb4, false, j, "acc_scale_in");
            add_span(v, d[j].acc_q_out, n, true, j, "acc_q_out");
            add_span(v, d[j].acc_scale_out, nb4, true, j, "acc_scale_out");
        }
        add_span(v, d[j].grad, n * 2, false, j, "grad_bf16");
    }
    return check_spans(v);
}

// ------------------------------------------------------------ chunk maps ----
//
// A launch reads its tensor list from two device tables: the descriptors (one per
// tensor: pointers, n, flags) and the chunk map (one (tensor, begin) entry per
// 8192-element chunk).  The chunk map depends only on the tensors' sizes, so it is
// built and uploaded once per size list and kept (immutable).  Descriptors change
// from call to call (every micro-step reads a different grad buffer, the slot pool
// hands out alternating slots), so they are staged per call through a ring buffer
// (below); steady-state calls allocate nothing and never synchronize.

struct ChunkMap {
    std::vector<int64_t> key;       // device, then the sizes
    Chunk* dev = nullptr;
    void* host = nullptr;           // pinned staging of the upload, kept with the entry
    int64_t n_chunks = 0;
    cudaEvent_t ready = nullptr;    // the upload is done
};

constexpr size_t kMaxMaps = 4096;

std::mutex g_mu;
std::unordered_multimap<uint64_t, ChunkMap*> g_maps;

uint64_t fnv1a(const void* data, size_t n) {
    const unsigned char* p = static_cast<const unsigned char*>(data);
    uint64_t h = 1469598103934665603ull;
    for (size_t i = 0; i < n; ++i) { h ^= p[i]; h *= 1099511628211ull; }
    return h;
}

void free_map(ChunkMap* m) {
    if (m->ready) cudaEventDestroy(m->ready);
    if (m->dev) cudaFree(m->dev);
    if (m->host) cudaFreeHost(m->host);
    delete m;
}

int get_chunk_map(int device, const std::vector<int64_t>& sizes, cudaStream_t stream,
                  ChunkMap** out) {
    std::vector<int64_t> key;
    key.reserve(sizes.size() + 1);
    key.push_back(device);
    key.insert(key.end(), sizes.begin(), sizes.end());
    const uint64_t h = fnv1a(key.data(), key.size() * sizeof(int64_t));
    auto range = g_maps.equal_range(h);
    for (auto it = range.first; it != range.second; ++it)
        if (it->second->key == key) { *out = it->second; return LEMA_OK; }

    int64_t n_chunks = 0;
    for (int64_t n : sizes) n_chunks += (n + kChunk - 1) / kChunk;
    if (n_chunks > int64_t(0x7FFFFFFF)) return set_error(LEMA_ERR_ARG, "too many elements for one launch");
    if (g_maps.size() >= kMaxMaps) {        // a pathological number of shapes: start over
        cudaDeviceSynchronize();
        for (auto& kv : g_maps) free_map(kv.second);
        g_maps.clear();
    }
    ChunkMap* m = new ChunkMap();
    m->key = std::move(key);
    m->n_chunks = n_chunks;
    cudaError_t e = cudaEventCreateWithFlags(&m->ready, cudaEventDisableTiming);
    if (e == cudaSuccess && n_chunks > 0) {
        const size_t bytes = sizeof(Chunk) * size_t(n_chunks);
        if ((e = cudaMalloc(&m->dev, bytes)) == cudaSuccess &&
            (e = cudaMallocHost(&m->host, bytes)) == cudaSuccess) {
            Chunk* c = static_cast<Chunk*>(m->host);
            int64_t i = 0;
            for (size_t j = 0; j < sizes.size(); ++j)
                for (int64_t b = 0; b < sizes[j]; b += kChunk) c[i++] = Chunk{int32_t(j), 0, b};
            e = cudaMemcpyAsync(m->dev, m->host, bytes, cudaMemcpyHostToDevice, stream);
        }
    }
    if (e == cudaSuccess) e = cudaEventRecord(m->ready, stream);
    if (e != cudaSuccess) {
        free_map(m);
        return cuda_error(e, "chunk map upload");
    }
    g_maps.emplace(h, m);
    *out = m;
    return LEMA_OK;
}

// -------------------------------------------------------- descriptor ring ----
//
// Per device: a device buffer and a pinned host buffer of the same size, used as a
// ring.  A call writes its descriptors into the next free region of the host
// buffer, enqueues a small kernel on its own stream that copies the region to the
// device (the SMs read pinned host memory directly, so the copy never waits behind
// bulk host<->device transfers on a copy engine), launches, and records an event;
// the region is reused only after that event (after the kernel that read it) has
// completed.  The host waits only if the whole ring is still in flight.

struct Ring {
    unsigned char* dev = nullptr;
    unsigned char* host = nullptr;
    size_t size = 0;
    size_t head = 0;
    struct Use {
        size_t off, len;
        cudaEvent_t ev;
    };
    std::deque<Use> inflight;
    std::vector<cudaEvent_t> spare;
};

constexpr size_t kRingBytes = size_t(4) << 20;
std::unordered_map<int, Ring*> g_rings;

int ring_drain(Ring* r) {
    while (!r->inflight.empty()) {
        cudaError_t e = cudaEventSynchronize(r->inflight.front().ev);
        if (e != cudaSuccess) return cuda_error(e, "descriptor ring");
        r->spare.push_back(r->inflight.front().ev);
        r->inflight.pop_front();
    }
    return LEMA_OK;
}

int ring_reserve(int device, size_t len, Ring** out, size_t* off) {
    Ring*& r = g_rings[device];
    if (!r) r = new Ring();
    len = (len + 255) & ~size_t(255);
    if (len > r->size) {                           // first use, or a larger tensor list
        int rc = ring_drain(r);
        if (rc != LEMA_OK) return rc;
        if (r->dev) cudaFree(r->dev);
        if (r->host) cudaFreeHost(r->host);
        r->dev = r->host = nullptr;
        r->size = 0;
        const size_t size = std::max(kRingBytes, 4 * len);
        cudaError_t e = cudaMalloc(&r->dev, size);
        if (e == cudaSuccess) e = cudaMallocHost(&r->host, size);
        if (e != cudaSuccess) return cuda_error(e, "descriptor ring allocation");
        r->size = size;
        r->head = 0;
    }
    if (r->head + len > r->size) r->head = 0;
    // In-flight regions form one circular run starting at the front; only its head
    // end can overlap the new region.
    while (!r->inflight.empty()) {
        const Ring::Use& u = r->inflight.front();
        const bool overlap = u.off < r->head + len && r->head < u.off + u.len;
        cudaError_t e = overlap ? cudaEventSynchronize(u.ev) : cudaEventQuery(u.ev);
        if (e == cudaErrorNotReady) break;
        if (e != cudaSuccess) return cuda_error(e, "descriptor ring");
        r->spare.push_back(u.ev);
        r->inflight.pop_front();
    }
    *out = r;
    *off = r->head;
    return LEMA_OK;
}

int ring_commit(Ring* r, size_t off, size_t len, cudaStream_t stream) {
    cudaEvent_t ev = nullptr;
    if (!r->spare.empty()) {
        ev = r->spare.back();
        r->spare.pop_back();
    } else {
        cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_error(e, "cudaEventCreate");
    }
    cudaError_t e = cudaEventRecord(ev, stream);
    if (e != cudaSuccess) return cuda_error(e, "cudaEventRecord");
    len = (len + 255) & ~size_t(255);
    r->inflight.push_back(Ring::Use{off, len, ev});
    r->head = off + len;
    return LEMA_OK;
}

// Validate, stage the descriptors, make the stream wait for the chunk map, then
// run `launch(device descriptors, chunk map, n_chunks)` and retire the region.
template <typename Desc, typename Launch>
int stage_and_launch(const Desc* descs, int32_t count, cudaStream_t stream, int verdict,
                     Launch launch, const char* what) {
    if (verdict != LEMA_OK) return verdict;
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
    std::vector<int64_t> sizes(static_cast<size_t>(count));
    for (int32_t j = 0; j < count; ++j) sizes[size_t(j)] = descs[j].n;
    ChunkMap* map = nullptr;
    int rc = get_chunk_map(device, sizes, stream, &map);
    if (rc != LEMA_OK || map->n_chunks == 0) return rc;
    Ring* r = nullptr;
    size_t off = 0;
    const size_t bytes = sizeof(Desc) * size_t(count);
    rc = ring_reserve(device, bytes, &r, &off);
    if (rc != LEMA_OK) return rc;
    std::memcpy(r->host + off, descs, bytes);
    if ((e = launch_install(r->dev + off, r->host + off, bytes, stream)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(stream, map->ready, 0)) != cudaSuccess)
        return cuda_error(e, "descriptor upload");
    e = launch(reinterpret_cast<const Desc*>(r->dev + off), map->dev, map->n_chunks);
    if (e != cudaSuccess) return cuda_error(e, what);
    return ring_commit(r, off, bytes, stream);
}

// Tables of at most kValueTableMax tensors go to the kernel by value, as a launch
// parameter: one launch per call, no upload.
template <typename Desc, typename Launch>
int launch_by_value(const Desc* descs, int32_t count, cudaStream_t stream, int verdict,
                    Launch launch, const char* what) {
    if (verdict != LEMA_OK) return verdict;
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
    std::vector<int64_t> sizes(static_cast<size_t>(count));
    for (int32_t j = 0; j < count; ++j) sizes[size_t(j)] = descs[j].n;
    ChunkMap* map = nullptr;
    const int rc = get_chunk_map(device, sizes, stream, &map);
    if (rc != LEMA_OK || map->n_chunks == 0) return rc;
    if ((e = cudaStreamWaitEvent(stream, map->ready, 0)) != cudaSuccess)
        return cuda_error(e, "chunk map upload");
    e = launch(descs, map->dev, map->n_chunks);
    return e == cudaSuccess ? LEMA_OK : cuda_error(e, what);
}

}  // namespace

int run_accum(const AccDesc* descs, int32_t count, cudaStream_t stream, bool pdl) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (count <= kValueTableMax)
        return launch_by_value(
            descs, count, stream, validate_accum(descs, count),
            [&](const AccDesc* d, const Chunk* c, int64_t n) {
                return launch_accum_v(d, count, c, n, stream, pdl);
            },
            "accum_grad launch");
    return stage_and_launch(
        descs, count, stream, validate_accum(descs, count),
        [&](const AccDesc* d, const Chunk* c, int64_t n) {
            return launch_accum(d, c, n, stream, pdl);
        },
        "accum_grad launch");
}

int run_step(const StepDesc* descs, int32_t count, const StepScalars& s, cudaStream_t stream,
             bool pdl) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (count <= kValueTableMax)
        return launch_by_value(
            descs, count, stream, validate_step(descs, count),
            [&](const StepDesc* d, const Chunk* c, int64_t n) {
                return launch_step_v(d, count, c, n, s, stream, pdl);
            },
            "adamw step launch");
    return stage_and_launch(
        descs, count, stream, validate_step(descs, count),
        [&](const StepDesc* d, const Chunk* c, int64_t n) {
            return launch_step(d, c, n, s, stream, pdl);
        },
        "adamw step launch");
}

int run_merge(const MergeDesc* descs, int32_t count, cudaStream_t stream) {
    std::lock_guard<std::mutex> lock(g_mu);
    return stage_and_launch(
        descs, count, stream, validate_merge(descs, count),
        [&](const MergeDesc* d, const Chunk* c, int64_t n) { return launch_merge(d, c, n, stream); },
        "merge launch");
}

int run_accum_q8(const AccDescQ8* descs, int32_t count, cudaStream_t stream) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (count <= kValueTableMax)
        return launch_by_value(
            descs, count, stream, validate_accum_q8(descs, count),
            [&](const AccDescQ8* d, const Chunk* c, int64_t n) {
                return launch_accum_q8_v(d, count, c, n, stream);
            },
            "8-bit accumulate launch");
    return stage_and_launch(
        descs, count, stream, validate_accum_q8(descs, count),
        [&](const AccDescQ8* d, const Chunk* c, int64_t n) { return launch_accum_q8(d, c, n, stream); },
        "8-bit accumulate launch");
}

int run_step_q8(const StepDescQ8* descs, int32_t count, const StepScalars& s, cudaStream_t stream,
                unsigned int* gave_up) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (count <= kValueTableMax)
        return launch_by_value(
            descs, count, stream, validate_step_q8(descs, count),
            [&](const StepDescQ8* d, const Chunk* c, int64_t n) {
                return launch_step_q8_v(d, count, c, n, s, gave_up, stream);
            },
            "8-bit adamw step launch");
    return stage_and_launch(
        descs, count, stream, validate_step_q8(descs, count),
        [&](const StepDescQ8* d, const Chunk* c, int64_t n) {
            return launch_step_q8(d, c, n, s, gave_up, stream);
        },
        "8-bit adamw step launch");
}

// ------------------------------------------------- kernel give-up reporting ----

int gave_up_flag_alloc(GaveUpFlag* f) {
    void* h = nullptr;
    cudaError_t e = cudaHostAlloc(&h, 64, cudaHostAllocMapped | cudaHostAllocPortable);
    if (e != cudaSuccess) return cuda_error(e, "cudaHostAlloc (kernel status word)");
    std::memset(h, 0, 64);
    void* d = nullptr;
    e = cudaHostGetDevicePointer(&d, h, 0);
    if (e != cudaSuccess) {
        cudaFreeHost(h);
        return cuda_error(e, "cudaHostGetDevicePointer (kernel status word)");
    }
    f->host = static_cast<volatile unsigned int*>(h);
    f->dev = static_cast<unsigned int*>(d);
    return LEMA_OK;
}

void gave_up_flag_free(GaveUpFlag* f) {
    if (f->host) cudaFreeHost(const_cast<unsigned int*>(f->host));
    f->host = nullptr;
    f->dev = nullptr;
}

int gave_up_take(const GaveUpFlag& f, const char* where) {
    if (!f.host) return LEMA_OK;
    // An atomic exchange, so that a kernel still running that sets the word between
    // a read and a reset on the host is not lost: its 1 stays for the next check.
    const unsigned int was =
        __atomic_exchange_n(const_cast<unsigned int*>(f.host), 0u, __ATOMIC_ACQ_REL);
    if (was == 0u) return LEMA_OK;
    return set_error(LEMA_ERR_TIMEOUT,
                     "%s: an 8-bit step kernel gave up waiting for its staged inputs (see "
                     "lema_kernel_wait_timeouts); the groups it had not finished kept their old "
                     "outputs, so that step's results are incomplete",
                     where);
}

namespace {

// The flag of the direct 8-bit step calls, one per device (allocated on first use).
int direct_flag(GaveUpFlag** out) {
    constexpr int kMaxDevices = 64;
    static GaveUpFlag flags[kMaxDevices];
    static std::mutex mu;
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices)
        return set_error(LEMA_ERR_STATE, "device %d is beyond the %d devices supported", dev,
                         kMaxDevices);
    std::lock_guard<std::mutex> g(mu);
    if (!flags[dev].host) {
        const int rc = gave_up_flag_alloc(&flags[dev]);
        if (rc != LEMA_OK) return rc;
    }
    *out = &flags[dev];
    return LEMA_OK;
}

}  // namespace

}  // namespace lema

// =================================================================== C ABI ====

using namespace lema;

extern "C" const char* lema_last_error(void) { return g_err; }

extern "C" int lema_test_divide_by_constant(const float* divisors, int32_t count,
                                            int64_t* mismatches, int64_t* outside) {
    g_err[0] = '\0';
    if (count < 0 || (count > 0 && (!divisors || !mismatches || !outside)))
        return set_error(LEMA_ERR_ARG, "bad arguments");
    for (int32_t i = 0; i < count; ++i)
        if (!(divisors[i] > 0x1p-27f && divisors[i] <= 1.0f))
            return set_error(LEMA_ERR_ARG, "divisor %d is outside (2^-27, 1]", i);
    unsigned long long* bad = nullptr;
    cudaError_t e = cudaMalloc(&bad, 2 * sizeof(unsigned long long) * size_t(count > 0 ? count : 1));
    if (e != cudaSuccess) return cuda_error(e, "cudaMalloc");
    e = cudaMemset(bad, 0, 2 * sizeof(unsigned long long) * size_t(count > 0 ? count : 1));
    for (int32_t i = 0; i < count && e == cudaSuccess; ++i)
        e = check_div_by_const(divisors[i], rcp_rn(divisors[i]), bad + 2 * i, nullptr);
    std::vector<unsigned long long> h(2 * size_t(count > 0 ? count : 1));
    if (e == cudaSuccess)
        e = cudaMemcpy(h.data(), bad, h.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
    cudaFree(bad);
    if (e != cudaSuccess) return cuda_error(e, "division check");
    for (int32_t i = 0; i < count; ++i) {
        mismatches[i] = int64_t(h[2 * size_t(i)]);
        outside[i] = int64_t(h[2 * size_t(i) + 1]);
    }
    return LEMA_OK;
}

extern "C" int lema_test_kernel_wait_limit(int64_t limit_ns) {
    g_err[0] = '\0';
    const cudaError_t e = set_wait_limit(limit_ns);
    return e == cudaSuccess ? LEMA_OK : cuda_error(e, "setting the kernel wait limit");
}

extern "C" int lema_kernel_wait_timeouts(int64_t* count) {
    g_err[0] = '\0';
    if (!count) return set_error(LEMA_ERR_ARG, "count is NULL");
    unsigned long long n = 0;
    const cudaError_t e = read_wait_timeouts(&n);
    if (e != cudaSuccess) return cuda_error(e, "reading the kernel wait counter");
    *count = int64_t(n);
    return LEMA_OK;
}

extern "C" const char* lema_status_string(int status) {
    switch (status) {
        case LEMA_OK: return "LEMA_OK";
        case LEMA_ERR_ARG: return "LEMA_ERR_ARG";
        case LEMA_ERR_ALIGN: return "LEMA_ERR_ALIGN";
        case LEMA_ERR_CUDA: return "LEMA_ERR_CUDA";
        case LEMA_ERR_OOM: return "LEMA_ERR_OOM";
        case LEMA_ERR_TIMEOUT: return "LEMA_ERR_TIMEOUT";
        case LEMA_ERR_STATE: return "LEMA_ERR_STATE";
        case LEMA_ERR_IO: return "LEMA_ERR_IO";
        default: return "LEMA_ERR_UNKNOWN";
    }
}

extern "C" int lema_accum_grad(const lema_grad* grads, int32_t count, void* cuda_stream) {
    g_err[0] = '\0';
    if (count < 0) return set_error(LEMA_ERR_ARG, "count must be >= 0 (got %d)", count);
    if (count == 0) return LEMA_OK;
    if (!grads) return set_error(LEMA_ERR_ARG, "grads is NULL");
    std::vector<AccDesc> d(static_cast<size_t>(count));
    for (int32_t j = 0; j < count; ++j) {
        const lema_grad& g = grads[j];
        if (g.n < 0) return set_error(LEMA_ERR_ARG, "tensor %d: n must be >= 0", j);
        if ((g.flags & ~int32_t(LEMA_GRAD_FIRST)) != 0 || g.reserved != 0)
            return set_error(LEMA_ERR_ARG, "tensor %d: unknown flags", j);
        if (g.n > 0) {
            if (!g.acc || !g.grad_bf16)
                return set_error(LEMA_ERR_ARG, "tensor %d: NULL acc or grad_bf16", j);
            if (!aligned16(g.acc) || !aligned16(g.grad_bf16))
                return set_error(LEMA_ERR_ALIGN, "tensor %d: base address not 16-byte aligned", j);
        }
        const bool first = (g.flags & LEMA_GRAD_FIRST) != 0;
        d[j] = AccDesc{first ? nullptr : g.acc, g.acc, g.grad_bf16, g.n};
    }
    return run_accum(d.data(), count, static_cast<cudaStream_t>(cuda_stream), true);
}

extern "C" int lema_adamw_step(const lema_tensor* tensors, int32_t count, int64_t step, double lr,
                               double beta1, double beta2, double eps, double weight_decay,
                               int32_t accum_steps, void* cuda_stream) {
    g_err[0] = '\0';
    StepScalars s;
    int rc = make_scalars(step, lr, beta1, beta2, eps, weight_decay, accum_steps, &s);
    if (rc != LEMA_OK) return rc;
    if (count < 0) return set_error(LEMA_ERR_ARG, "count must be >= 0 (got %d)", count);
    if (count == 0) return LEMA_OK;
    if (!tensors) return set_error(LEMA_ERR_ARG, "tensors is NULL");
    std::vector<StepDesc> d(static_cast<size_t>(count));
    for (int32_t j = 0; j < count; ++j) {
        const lema_tensor& t = tensors[j];
        if (t.n < 0) return set_error(LEMA_ERR_ARG, "tensor %d: n must be >= 0", j);
        if ((t.flags & ~int32_t(LEMA_STEP_KEEP_ACC)) != 0 || t.reserved != 0)
            return set_error(LEMA_ERR_ARG, "tensor %d: unknown flags", j);
        const int outs = (t.master_out != nullptr) + (t.m_out != nullptr) + (t.v_out != nullptr);
        if (outs != 0 && outs != 3)
            return set_error(LEMA_ERR_ARG,
                             "tensor %d: master_out, m_out, v_out must be all NULL or all set", j);
        const bool in_place = outs == 0;
        if (t.n > 0 && !t.acc && !t.grad_bf16)
            return set_error(LEMA_ERR_ARG, "tensor %d: acc may be NULL only with grad_bf16", j);
        if (t.n > 0 && !t.acc && accum_steps != 1)
            return set_error(LEMA_ERR_ARG, "tensor %d: acc may be NULL only when accum_steps == 1",
                             j);
        StepDesc& x = d[j];
        x.master_in = t.master;
        x.m_in = t.m;
        x.v_in = t.v;
        x.acc = t.acc;
        x.orig = t.orig_bf16;
        x.master_out = in_place ? t.master : t.master_out;
        x.m_out = in_place ? t.m : t.m_out;
        x.v_out = in_place ? t.v : t.v_out;
        x.delta = t.delta;
        x.w = t.w_bf16;
        x.grad = t.grad_bf16;
        x.n = t.n;
        x.flags = (in_place && t.acc && !(t.flags & LEMA_STEP_KEEP_ACC)) ? kZeroAcc : 0;
        if (t.n == 0) continue;
        const void* ptrs[] = {x.master_in, x.m_in, x.v_in, x.orig, x.master_out,
                              x.m_out, x.v_out, x.delta, x.w};
        for (const void* p : ptrs)
            if (!p) return set_error(LEMA_ERR_ARG, "tensor %d: NULL buffer", j);
        const void* any[] = {x.master_in, x.m_in, x.v_in, x.acc, x.orig, x.master_out,
                             x.m_out, x.v_out, x.delta, x.w, x.grad};
        for (const void* p : any)
            if (p && !aligned16(p))
                return set_error(LEMA_ERR_ALIGN, "tensor %d: base address not 16-byte aligned", j);
    }
    return run_step(d.data(), count, s, static_cast<cudaStream_t>(cuda_stream), true);
}

extern "C" int lema_accum_grad_q8(const lema_grad_q8* grads, int32_t count, void* cuda_stream) {
    g_err[0] = '\0';
    if (count < 0) return set_error(LEMA_ERR_ARG, "count must be >= 0 (got %d)", count);
    if (count == 0) return LEMA_OK;
    if (!grads) return set_error(LEMA_ERR_ARG, "grads is NULL");
    std::vector<AccDescQ8> d(static_cast<size_t>(count));
    for (int32_t j = 0; j < count; ++j) {
        const lema_grad_q8& g = grads[j];
        if (g.n < 0) return set_error(LEMA_ERR_ARG, "tensor %d: n must be >= 0", j);
        if ((g.flags & ~int32_t(LEMA_GRAD_FIRST)) != 0 || g.reserved != 0)
            return set_error(LEMA_ERR_ARG, "tensor %d: unknown flags", j);
        if (g.n > 0) {
            if (!g.acc_q || !g.acc_scale || !g.grad_bf16)
                return set_error(LEMA_ERR_ARG, "tensor %d: NULL acc_q, acc_scale or grad_bf16", j);
            if (!aligned16(g.acc_q) || !aligned16(g.acc_scale) || !aligned16(g.grad_bf16))
                return set_error(LEMA_ERR_ALIGN, "tensor %d: base address not 16-byte aligned", j);
        }
        const bool first = (g.flags & LEMA_GRAD_FIRST) != 0;
        d[j] = AccDescQ8{first ? nullptr : g.acc_q, first ? nullptr : g.acc_scale, g.acc_q,
                         g.acc_scale, g.grad_bf16, g.n};
    }
    return run_accum_q8(d.data(), count, static_cast<cudaStream_t>(cuda_stream));
}

extern "C" int lema_adamw_step_q8(const lema_tensor_q8* tensors, int32_t count, int64_t step,
                                  double lr, double beta1, double beta2, double eps,
                                  double weight_decay, int32_t accum_steps, void* cuda_stream) {
    g_err[0] = '\0';
    StepScalars s;
    int rc = make_scalars(step, lr, beta1, beta2, eps, weight_decay, accum_steps, &s);
    if (rc != LEMA_OK) return rc;
    if (count < 0) return set_error(LEMA_ERR_ARG, "count must be >= 0 (got %d)", count);
    if (count == 0) return LEMA_OK;
    if (!tensors) return set_error(LEMA_ERR_ARG, "tensors is NULL");
    std::vector<StepDescQ8> d(static_cast<size_t>(count));
    for (int32_t j = 0; j < count; ++j) {
        const lema_tensor_q8& t = tensors[j];
        if (t.n < 0) return set_error(LEMA_ERR_ARG, "tensor %d: n must be >= 0", j);
        if ((t.flags & ~int32_t(LEMA_STEP_KEEP_ACC)) != 0 || t.reserved != 0)
            return set_error(LEMA_ERR_ARG, "tensor %d: unknown flags", j);
        const int outs = (t.master_out != nullptr) + (t.m_q_out != nullptr) +
                         (t.m_scale_out != nullptr) + (t.r_q_out != nullptr) +
                         (t.r_scale_out != nullptr);
        if (outs != 0 && outs != 5)
            return set_error(LEMA_ERR_ARG, "tensor %d: the five *_out fields must be all NULL or all set",
                             j);
        const bool in_place = outs == 0;
        const bool has_acc = t.acc_q != nullptr || t.acc_scale != nullptr;
        if (t.n > 0 && has_acc && (!t.acc_q || !t.acc_scale))
            return set_error(LEMA_ERR_ARG, "tensor %d: acc_q and acc_scale go together", j);
        if (t.n > 0 && !has_acc && (!t.grad_bf16 || accum_steps != 1))
            return set_error(LEMA_ERR_ARG,
                             "tensor %d: the accumulator may be NULL only with grad_bf16 and accum_steps == 1",
                             j);
        StepDescQ8& x = d[j];
        x.master_in = t.master;
        x.m_q_in = t.m_q;
        x.m_scale_in = t.m_scale;
        x.r_q_in = t.r_q;
        x.r_scale_in = t.r_scale;
        x.acc_q = t.acc_q;
        x.acc_scale = t.acc_scale;
        x.grad = t.grad_bf16;
        x.orig = t.orig_bf16;
        x.master_out = in_place ? t.master : t.master_out;
        x.m_q_out = in_place ? t.m_q : t.m_q_out;
        x.m_scale_out = in_place ? t.m_scale : t.m_scale_out;
        x.r_q_out = in_place ? t.r_q : t.r_q_out;
        x.r_scale_out = in_place ? t.r_scale : t.r_scale_out;
        x.delta = t.delta;
        x.w = t.w_bf16;
        x.n = t.n;
        x.flags = (in_place && has_acc && !(t.flags & LEMA_STEP_KEEP_ACC)) ? kZeroAcc : 0;
        if (t.n == 0) continue;
        const void* need[] = {x.master_in, x.m_q_in, x.m_scale_in, x.r_q_in, x.r_scale_in,
                              x.orig, x.master_out, x.m_q_out, x.m_scale_out, x.r_q_out,
                              x.r_scale_out, x.delta, x.w};
        for (const void* p : need)
            if (!p) return set_error(LEMA_ERR_ARG, "tensor %d: NULL buffer", j);
        const void* any[] = {x.master_in, x.m_q_in, x.m_scale_in, x.r_q_in, x.r_scale_in,
                             x.acc_q, x.acc_scale, x.grad, x.orig, x.master_out, x.m_q_out,
                             x.m_scale_out, x.r_q_out, x.r_scale_out, x.delta, x.w};
        for (const void* p : any)
            if (p && !aligned16(p))
                return set_error(LEMA_ERR_ALIGN, "tensor %d: base address not 16-byte aligned", j);
    }
    GaveUpFlag* flag = nullptr;
    rc = direct_flag(&flag);
    if (rc != LEMA_OK) return rc;
    rc = gave_up_take(*flag, "lema_adamw_step_q8 (an earlier call; nothing was launched now)");
    if (rc != LEMA_OK) return rc;
    return run_step_q8(d.data(), count, s, static_cast<cudaStream_t>(cuda_stream), flag->dev);
}

extern "C" int lema_merge_delta(const lema_merge* items, int32_t count, void* cuda_stream) {
    g_err[0] = '\0';
    if (count < 0) return set_error(LEMA_ERR_ARG, "count must be >= 0 (got %d)", count);
    if (count == 0) return LEMA_OK;
    if (!items) return set_error(LEMA_ERR_ARG, "items is NULL");
    std::vector<MergeDesc> d(static_cast<size_t>(count));
    for (int32_t j = 0; j < count; ++j) {
        const lema_merge& m = items[j];
        if (m.n < 0) return set_error(LEMA_ERR_ARG, "tensor %d: n must be >= 0", j);
        if (m.n > 0) {
            if (!m.base_bf16 || !m.delta || !m.merged_bf16)
                return set_error(LEMA_ERR_ARG, "tensor %d: NULL buffer", j);
            if (!aligned16(m.base_bf16) || !aligned16(m.delta) || !aligned16(m.merged_bf16))
                return set_error(LEMA_ERR_ALIGN, "tensor %d: base address not 16-byte aligned", j);
        }
        d[j] = MergeDesc{m.base_bf16, m.delta, m.merged_bf16, m.n};
    }
    return run_merge(d.data(), count, static_cast<cudaStream_t>(cuda_stream));
}
