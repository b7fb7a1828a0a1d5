// Host side of the C ABI declared in include/kvm.h: argument validation,
// workspace layout, the data-independent growth schedule, RoPE tables and
// kernel launches.  Nothing here touches tensor data on the host.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/kvm.h"
#include "kvm_host.h"
#include "kvm_internal.cuh"

using kvm::D;

namespace {
// NVTX range over an entry point (a no-op unless a profiler is attached)
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};
}  // namespace
using kvm::Sched;

namespace kvm {
namespace host {
thread_local std::string g_err = "no error";
}  // namespace host
}  // namespace kvm

using kvm::host::ALIGN;
using kvm::host::g_err;
using kvm::host::Layout;

namespace kvm {
namespace host {

size_t align_up(size_t x) { return (x + ALIGN - 1) / ALIGN * ALIGN; }

int64_t n_events_for(const kvm_config& c, int64_t N) {
    const int64_t nchunks = (N + c.chunk - 1) / c.chunk;
    const int64_t e = nchunks - c.window / c.chunk - 1;
    return e > 0 ? e : 0;
}

// Capacity after t overflowed tokens ("Key-Value Means", technical summary,
// Core mechanism 3: fixed-size or power-law growth), in double precision.
int64_t capacity(const kvm_config& c, int64_t t) {
    if (c.sched == KVM_SCHED_FIXED) return c.max_slots;
    if (t <= 0) return c.n_sinks;
    return (int64_t)c.n_sinks + (int64_t)std::ceil((double)c.coef * std::pow((double)t, (double)c.expo));
}

// One fold event's slot bookkeeping from the slot count n and overflow count t before it.
Sched event_sched(const kvm_config& c, int64_t first_pos, int64_t n, int64_t t) {
    Sched s;
    int64_t sinks = 0;
    for (int64_t i = 0; i < c.chunk; ++i) sinks += (first_pos + i < c.n_sinks);
    const int64_t n0 = n + sinks;
    const int64_t ncand = c.chunk - sinks;
    int64_t a = capacity(c, t + c.chunk) - n0;
    if (a < 0) a = 0;
    if (a > ncand) a = ncand;
    s.n_before = (int)n;
    s.n0 = (int)n0;
    s.a = (int)a;
    s.n_after = (int)(n0 + a);
    return s;
}

bool validate(const kvm_config* c, std::string& why) {
    if (!c) { why = "config is NULL"; return false; }
    if (c->batch < 1 || c->heads < 1) { why = "batch and heads must be >= 1"; return false; }
    if (c->head_dim != D) { why = "head_dim must be 64 (the only head size this library supports)"; return false; }
    if (c->rope_dims < 0 || c->rope_dims > c->head_dim || (c->rope_dims & 1)) {
        why = "rope_dims must be even and in [0, head_dim]"; return false;
    }
    if (!(c->rope_theta > 0.0f)) { why = "rope_theta must be > 0"; return false; }
    if (c->chunk < 16 || c->chunk > 256 || c->chunk % 16) {
        why = "chunk must be a multiple of 16 in [16, 256]"; return false;
    }
    if (c->window < 0 || c->window % c->chunk) { why = "window must be a non-negative multiple of chunk"; return false; }
    if (c->n_sinks < 0 || c->n_sinks > c->chunk) { why = "n_sinks must be in [0, chunk]"; return false; }
    if (c->max_slots < c->n_sinks + 1 || c->max_slots > 4096) {
        why = "max_slots must be in [n_sinks + 1, 4096]"; return false;
    }
    if (c->sched != KVM_SCHED_FIXED && c->sched != KVM_SCHED_POWER) { why = "unknown schedule"; return false; }
    if (c->sched == KVM_SCHED_POWER && (!(c->coef > 0.0f) || !(c->expo > 0.0f) || c->expo > 1.0f)) {
        why = "power schedule needs coef > 0 and 0 < expo <= 1"; return false;
    }
    if (!(c->ln_eps > 0.0f)) { why = "ln_eps must be > 0"; return false; }
    if (c->dtype != KVM_BF16 && c->dtype != KVM_FP32) { why = "unknown dtype"; return false; }
    if (c->max_tokens < 1 || c->max_tokens > (1 << 22)) { why = "max_tokens must be in [1, 2^22]"; return false; }
    if (c->flags & ~KVM_FLAG_NO_VALUE_NORM) { why = "unknown flags"; return false; }
    return true;
}

Layout layout_of(const kvm_config& c) {
    Layout L;
    const size_t BH = (size_t)c.batch * c.heads, M = c.max_slots, d = D;
    const size_t es = c.dtype == KVM_BF16 ? 2 : 4;
    const size_t ring = (size_t)c.window + c.chunk;
    const size_t E = (size_t)n_events_for(c, c.max_tokens);
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes); return at; };
    L.sum_k = take(BH * M * d * 4);
    L.sum_v = take(BH * M * d * 4);
    L.counts = take(BH * M * 4);
    L.rho = take(BH * M * 4);
    L.simdir = take(BH * M * d * 4);
    L.view_k = take(BH * M * (size_t)kvm::view_k_dims(c.rope_dims) * es);  // non-rotary dims only
    L.view_v = take(BH * M * d * es);
    L.ring_k = take(BH * ring * d * es);
    L.ring_v = take(BH * ring * d * es);
    L.ring_g = take(BH * ring * 4);
    L.ring_kr = take(BH * ring * d * es);
    L.snap_k = take(BH * E * M * d * es);
    L.snap_v = take(BH * E * M * d * es);
    L.rope = take((size_t)c.max_tokens * (c.rope_dims / 2) * sizeof(float2) + 16);
    L.sched = take((E + 1) * sizeof(Sched));
    L.status = take(256);  // status word at 0, attention tile-range counters at TILE_CTR_OFF
    L.k_rot = take(c.dtype == KVM_BF16 && c.rope_dims > 0 ? BH * (size_t)c.max_tokens * d * es : 0);
    L.q_rot = take(c.dtype == KVM_BF16 && c.rope_dims > 0 ? BH * (size_t)c.max_tokens * d * es : 0);
    L.has_lse = c.dtype == KVM_BF16 && c.chunk % 128 == 0;
    L.lse = take(L.has_lse ? BH * (size_t)c.max_tokens * 4 : 0);
    // the streamed-state chain's per-event log of touched rows (snapshots are rebuilt from it)
    kvm::FoldArgs probe{};
    probe.C = c.chunk;
    probe.M = c.max_slots;
    const bool logs = kvm::fold_logs_rows(probe, c.dtype == KVM_BF16);
    const size_t lrows = logs ? BH * E * (size_t)c.chunk : 0;
    L.log_k = take(lrows * d * es);
    L.log_v = take(lrows * d * es);
    L.log_idx = take(lrows * 4);
    L.log_cnt = take(logs ? BH * E * 4 : 0);
    L.logs = logs;
    L.total = o;
    return L;
}

}  // namespace host

namespace {
struct RopeFreqs {
    int half;
    double f[32];  // theta^(-2i/r), computed on the host in double
};

// cos/sin of p * theta^(-2i/r), evaluated in double precision, stored as float2
__global__ void rope_table_kernel(const RopeFreqs fr, int64_t n_pos, float2* out) {
    const int64_t total = n_pos * fr.half;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t p = i / fr.half;
        const int x = (int)(i % fr.half);
        const double ang = (double)p * fr.f[x];
        out[i] = make_float2((float)cos(ang), (float)sin(ang));
    }
}
}  // namespace

cudaError_t launch_rope_table(int rope_dims, float rope_theta, int64_t n_pos, float2* out, cudaStream_t s) {
    RopeFreqs fr;
    fr.half = rope_dims / 2;
    if (fr.half <= 0 || n_pos <= 0) return cudaSuccess;
    if (fr.half > 32) return cudaErrorInvalidValue;
    for (int i = 0; i < fr.half; ++i) fr.f[i] = std::pow((double)rope_theta, -2.0 * i / (double)rope_dims);
    const int64_t total = n_pos * fr.half;
    const int blocks = (int)((total + 255) / 256 < 1024 ? (total + 255) / 256 : 1024);
    rope_table_kernel<<<blocks, 256, 0, s>>>(fr, n_pos, out);
    return cudaGetLastError();
}

}  // namespace kvm

using kvm::host::capacity;
using kvm::host::event_sched;
using kvm::host::layout_of;
using kvm::host::n_events_for;
using kvm::host::validate;

namespace {

struct DeviceGuard {
    int prev = -1;
    explicit DeviceGuard(int dev) {
        cudaGetDevice(&prev);
        if (prev != dev) cudaSetDevice(dev);
    }
    ~DeviceGuard() {
        int cur = -1;
        cudaGetDevice(&cur);
        if (prev >= 0 && cur != prev) cudaSetDevice(prev);
    }
};

}  // namespace

struct kvm_layer {
    kvm_config cfg;
    char* ws;
    size_t ws_bytes;
    Layout L;
    int device;
    int64_t n_slots, n_overflow, pos;
    int64_t E_max;
    bool lse_valid = false;    // the last prefill wrote every query's log2-sum-exp (L.lse)
    int nsm = 0;               // SMs of the device
    std::vector<Sched> sched;  // prefill-from-empty schedule (host copy)
    cudaStream_t last_stream;
    std::string err;
    // optional per-kernel timing (kvm_layer_set_timing)
    struct Timed { int phase; cudaEvent_t a, b; };
    bool timing = false;
    std::vector<Timed> pool;
    size_t used = 0;
    double acc_ms[5] = {0, 0, 0, 0, 0};
    int64_t acc_n[5] = {0, 0, 0, 0, 0};
    int64_t kernels = 0;
    // overlapped prefill (kvm_layer_set_overlap)
    int overlap_segs = -1;
    int last_segs = 0;
    bool part_tried = false;
    kvm::host::Partition part;
    std::string part_why;
    ~kvm_layer() {
        for (auto& t : pool) {
            cudaEventDestroy(t.a);
            cudaEventDestroy(t.b);
        }
        if (part.ok) kvm::host::partition_free(&part);
    }

    template <typename P> P* at(size_t off) const { return reinterpret_cast<P*>(ws + off); }
    kvm_status fail(kvm_status st, const std::string& why) {
        err = why;
        return st;
    }
    kvm_status cuda_fail(cudaError_t e, const char* where) {
        err = std::string(where) + ": " + cudaGetErrorString(e);
        return KVM_ERR_CUDA;
    }
};

enum { PH_FOLD = 0, PH_ATTN = 1, PH_DECODE = 2, PH_OTHER = 3, PH_PROJ = 4 };

// Launch through f(), bracketed by timing events on s when timing is on.
template <class F>
static cudaError_t timed(kvm_layer* ly, int phase, cudaStream_t s, F&& f) {
    if (!ly->timing) return f();
    if (ly->used == ly->pool.size()) {
        kvm_layer::Timed t{phase, nullptr, nullptr};
        cudaError_t e = cudaEventCreate(&t.a);
        if (e == cudaSuccess) e = cudaEventCreate(&t.b);
        if (e != cudaSuccess) return e;
        ly->pool.push_back(t);
    }
    // copies of the handles: f() may launch through timed() again, and the pool's
    // storage moves when it grows
    kvm_layer::Timed& t = ly->pool[ly->used++];
    t.phase = phase;
    const cudaEvent_t ta = t.a, tb = t.b;
    cudaError_t e = cudaEventRecord(ta, s);
    if (e == cudaSuccess) e = f();
    const cudaError_t e2 = cudaEventRecord(tb, s);
    return e != cudaSuccess ? e : e2;
}

extern "C" {

size_t kvm_workspace_bytes(const kvm_config* cfg) {
    std::string why;
    if (!validate(cfg, why)) {
        g_err = why;
        return 0;
    }
    return layout_of(*cfg).total;
}

kvm_status kvm_layer_create(const kvm_config* cfg, void* dev_workspace, size_t bytes, kvm_layer** out) {
    NvtxRange nvtx_range("kvm_layer_create");
    std::string why;
    if (!out) { g_err = "out is NULL"; return KVM_ERR_INVALID_ARG; }
    *out = nullptr;
    if (!validate(cfg, why)) { g_err = why; return KVM_ERR_INVALID_ARG; }
    const Layout L = layout_of(*cfg);
    if (!dev_workspace || bytes < L.total) { g_err = "workspace missing or smaller than kvm_workspace_bytes"; return KVM_ERR_WORKSPACE; }
    if (reinterpret_cast<uintptr_t>(dev_workspace) % ALIGN) { g_err = "workspace must be 256-byte aligned"; return KVM_ERR_WORKSPACE; }
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, dev_workspace);
    if (e != cudaSuccess || attr.type != cudaMemoryTypeDevice) {
        cudaGetLastError();
        g_err = "workspace is not device memory";
        return KVM_ERR_WORKSPACE;
    }
    kvm_layer* ly = new kvm_layer();
    ly->cfg = *cfg;
    ly->ws = static_cast<char*>(dev_workspace);
    ly->ws_bytes = bytes;
    ly->L = L;
    ly->device = attr.device;
    ly->n_slots = ly->n_overflow = ly->pos = 0;
    ly->lse_valid = false;
    ly->E_max = n_events_for(*cfg, cfg->max_tokens);
    ly->last_stream = nullptr;
    DeviceGuard g(ly->device);
    cudaDeviceGetAttribute(&ly->nsm, cudaDevAttrMultiProcessorCount, ly->device);
    if (ly->nsm <= 0) ly->nsm = 1;
    // growth schedule of a prefill from the empty state
    ly->sched.resize((size_t)ly->E_max + 1);
    int64_t n = 0, t = 0;
    for (int64_t ev = 0; ev < ly->E_max; ++ev) {
        ly->sched[ev] = event_sched(*cfg, ev * cfg->chunk, n, t);
        n = ly->sched[ev].n_after;
        t += cfg->chunk;
    }
    // RoPE table: angle p * theta^(-2i/r) for pair i, computed in double on the device
    e = kvm::launch_rope_table(cfg->rope_dims, cfg->rope_theta, cfg->max_tokens,
                               reinterpret_cast<float2*>(ly->ws + L.rope), nullptr);
    if (e == cudaSuccess) e = cudaStreamSynchronize(nullptr);
    if (e == cudaSuccess)
        e = cudaMemcpy(ly->ws + L.sched, ly->sched.data(), ly->sched.size() * sizeof(Sched),
                       cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMemset(ly->ws + L.status, 0, 16);
    if (e == cudaSuccess) e = cudaMemset(ly->ws + L.counts, 0, L.rho - L.counts);
    // snapshot rows beyond a snapshot's slot count are read (and masked) by the
    // tensor-core attention: keep them finite
    if (e == cudaSuccess && L.rope > L.snap_k) e = cudaMemset(ly->ws + L.snap_k, 0, L.rope - L.snap_k);
    if (e != cudaSuccess) {
        g_err = std::string("kvm_layer_create: ") + cudaGetErrorString(e);
        delete ly;
        return KVM_ERR_CUDA;
    }
    *out = ly;
    return KVM_OK;
}

kvm_status kvm_prefill(kvm_layer* ly, const void* q, const void* k, const void* v, const float* gate,
                       int64_t n_tokens, void* out, void* cuda_stream, const kvm_debug* dbg) {
    NvtxRange nvtx_range("kvm_prefill");
    if (!ly) { g_err = "layer is NULL"; return KVM_ERR_INVALID_ARG; }
    const kvm_config& c = ly->cfg;
    if (n_tokens < 0 || n_tokens > c.max_tokens)
        return ly->fail(KVM_ERR_INVALID_ARG, "n_tokens must be in [0, max_tokens]");
    if (n_tokens > 0 && (!q || !k || !v || !gate || !out))
        return ly->fail(KVM_ERR_INVALID_ARG, "q, k, v, gate and out must be non-NULL");
    const int64_t E = n_events_for(c, n_tokens);
    if (E > 0 && ly->sched[E - 1].n_after > c.max_slots)
        return ly->fail(KVM_ERR_CAPACITY, "growth schedule exceeds max_slots for this n_tokens");
    if (dbg && dbg->max_events < 0) return ly->fail(KVM_ERR_INVALID_ARG, "dbg->max_events < 0");
    DeviceGuard g(ly->device);
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    ly->last_stream = s;
    const bool bf16 = c.dtype == KVM_BF16;
    const int BH = c.batch * c.heads;
    const Layout& L = ly->L;
    cudaError_t e = cudaSuccess;

    kvm::FoldArgs fa{};
    fa.sum_k = ly->at<float>(L.sum_k);
    fa.sum_v = ly->at<float>(L.sum_v);
    fa.counts = ly->at<int>(L.counts);
    fa.rho = ly->at<float>(L.rho);
    fa.simdir = ly->at<float>(L.simdir);
    fa.view_k = ly->ws + L.view_k;
    fa.view_v = ly->ws + L.view_v;
    fa.M = c.max_slots;
    fa.C = c.chunk;
    fa.S = c.n_sinks;
    fa.r = c.rope_dims;
    fa.ln_eps = c.ln_eps;
    fa.no_vnorm = (c.flags & KVM_FLAG_NO_VALUE_NORM) != 0;
    fa.k_src = k;
    fa.v_src = v;
    fa.g_src = gate;
    fa.src_row = n_tokens;
    fa.src_len = INT64_MAX / 4;
    fa.e_begin = 0;
    fa.e_end = (int)E;
    fa.sched = ly->at<Sched>(L.sched);
    fa.snap_k = ly->ws + L.snap_k;
    fa.snap_v = ly->ws + L.snap_v;
    fa.snap_events = (int)ly->E_max;
    if (L.logs) {
        fa.log_k = ly->ws + L.log_k;
        fa.log_v = ly->ws + L.log_v;
        fa.log_idx = ly->at<int>(L.log_idx);
        fa.log_cnt = ly->at<int>(L.log_cnt);
    }
    kvm::SnapRebuildArgs rb{};
    rb.log_k = fa.log_k;
    rb.log_v = fa.log_v;
    rb.log_idx = fa.log_idx;
    rb.log_cnt = fa.log_cnt;
    rb.snap_k = fa.snap_k;
    rb.snap_v = fa.snap_v;
    rb.snap_events = fa.snap_events;
    rb.C = c.chunk;
    rb.M = c.max_slots;
    rb.BH = (int)BH;
    rb.sched = fa.sched;
    if (dbg) {
        fa.dbg_assign = dbg->assign;
        fa.dbg_kind = dbg->kind;
        fa.dbg_m = dbg->max_sim;
        fa.dbg_gap = dbg->gap;
        fa.dbg_events = (int)(dbg->max_events < E ? dbg->max_events : E);
        fa.test_stall = dbg->test_stall;
    }
    fa.status = ly->at<int>(L.status);
    fa.BH = BH;

    kvm::AttnArgs aa{};
    aa.q = q;
    aa.k = k;
    aa.v = v;
    aa.out = out;
    aa.N = n_tokens;
    aa.C = c.chunk;
    aa.W = c.window;
    aa.snap_k = ly->ws + L.snap_k;
    aa.snap_v = ly->ws + L.snap_v;
    aa.snap_events = (int)ly->E_max;
    aa.M = c.max_slots;
    aa.sched = ly->at<Sched>(L.sched);
    aa.rope = ly->at<float2>(L.rope);
    aa.r = c.rope_dims;
    aa.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
    aa.BH = BH;
    aa.status = ly->at<int>(L.status);
    // every query's log2-sum-exp, kept for the backward (the tensor-core attention only)
    aa.lse = L.has_lse && n_tokens > 0 && kvm::attn_tc_supported(aa, bf16) ? ly->at<float>(L.lse) : nullptr;
    ly->lse_valid = false;

    kvm::RingFillArgs ra{};
    ra.k = k;
    ra.v = v;
    ra.g = gate;
    ra.ring_k = ly->ws + L.ring_k;
    ra.ring_v = ly->ws + L.ring_v;
    ra.ring_g = ly->at<float>(L.ring_g);
    ra.ring_kr = ly->ws + L.ring_kr;
    ra.rope = ly->at<float2>(L.rope);
    ra.r = c.rope_dims;
    ra.N = n_tokens;
    ra.first = E * c.chunk;
    ra.L = c.window + c.chunk;
    ra.BH = BH;
    const bool ring_work = n_tokens > ra.first;

    // tensor-core attention: keys rotated once, before it, instead of per tile
    kvm::RopeKeysArgs ka{};
    ka.k = k;
    ka.k_rot = ly->ws + L.k_rot;
    ka.rope = ly->at<float2>(L.rope);
    ka.r = c.rope_dims;
    ka.N = n_tokens;
    ka.BH = BH;
    const bool pre_rotate = bf16 && c.rope_dims > 0 && n_tokens > 0 && kvm::attn_tc_supported(aa, bf16);
    if (pre_rotate) {
        aa.k_rot = ka.k_rot;
        // the queries are rotated in the same pass
        ka.q = q;
        ka.q_rot = ly->ws + L.q_rot;
        aa.q_rot = ka.q_rot;
        // 32 rotary dims: only they are rotated and stored (the attention reads the rest of
        // each row from q and k)
        ka.compact = c.rope_dims == 32;
        aa.rot_compact = ka.compact;
        // the window ring is filled in the same pass
        if (ring_work) {
            ka.v = v;
            ka.g = gate;
            ka.ring_k = ra.ring_k;
            ka.ring_v = ra.ring_v;
            ka.ring_g = ra.ring_g;
            ka.ring_kr = ra.ring_kr;
            ka.first = ra.first;
            ka.L = ra.L;
        }
    }

    // overlapped prefill: fold segments on one SM partition, the attention of
    // the chunks each segment has made ready on the other
    int segs = 0;
    if (ly->overlap_segs != 0 && !dbg && E >= 2 &&
        (kvm::fold_tc_supported(fa, bf16) || kvm::fold_big_supported(fa, bf16)) &&
        kvm::attn_tc_supported(aa, bf16)) {
        if (!ly->part_tried) {
            ly->part_tried = true;
            kvm::host::partition_make(ly->device, BH, &ly->part, ly->part_why);
        }
        if (ly->part.ok) {
            // automatic: restarts of the on-chip chain reload its state (2 segments measured
            // best); the streamed chain restarts for free (8)
            segs = ly->overlap_segs > 0 ? ly->overlap_segs : (kvm::fold_tc_supported(fa, bf16) ? 2 : 8);
            if (segs > kvm::host::Partition::MAX_SEGS) segs = kvm::host::Partition::MAX_SEGS;
            if (segs > E) segs = (int)E;
        }
    }
    ly->last_segs = segs;

    if (segs > 0) {
        kvm::host::Partition& P = ly->part;
        int* ctr = reinterpret_cast<int*>(ly->ws + L.status + kvm::host::TILE_CTR_OFF);
        const int64_t tph = (n_tokens + 127) / 128, Wc = c.window / c.chunk, tpc = c.chunk / 128;
        // tiles (all rows) of the chunks whose state is complete once events < e_done are folded
        auto ready = [&](int64_t e_done) {
            int64_t t = (e_done + Wc + 1) * tpc;
            return (int)((t < tph ? t : tph) * BH);
        };
        // segment boundaries (events): equal parts, except that with two segments the first
        // ends at 40% of the events — the attention partition's own work before the first
        // segment's chunks (the rotation, the chunks that need no fold) ends well before the
        // chain's middle, and a shorter first segment hands it those chunks sooner
        // (measured on the fixed 8k workload: 0.573 -> 0.561 ms a step)
        auto bnd = [&](int sg) -> int64_t {
            if (segs == 2 && sg == 1) return E * 2 / 5 > 0 ? E * 2 / 5 : 1;
            return E * sg / segs;
        };
        // range 0: chunks that need no fold; range k + 1: the chunks segment k makes ready
        aa.n_ranges = segs + 1;
        aa.range_end[0] = ready(0);
        for (int sg = 0; sg < segs; ++sg) aa.range_end[sg + 1] = ready(bnd(sg + 1));
        e = cudaMemsetAsync(ctr, 0, sizeof(int) * aa.n_ranges, s);
        if (e == cudaSuccess) e = cudaEventRecord(P.ev_fork, s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(P.s_fold, P.ev_fork, 0);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(P.s_attn, P.ev_fork, 0);
        if (e != cudaSuccess) return ly->cuda_fail(e, "overlap set-up");
        aa.tile_ctr = ctr;
        if (pre_rotate) {
            ka.grid = 8 * P.sm_attn;
            e = timed(ly, PH_OTHER, P.s_attn, [&] { return kvm::launch_rope_keys(ka, P.s_attn); });
            if (e != cudaSuccess) return ly->cuda_fail(e, "key rotation launch");
            ly->kernels += 1;
            // the last attention launch (on s) reads the rotated keys as well
            e = cudaEventRecord(P.ev_attn, P.s_attn);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(s, P.ev_attn, 0);
            if (e != cudaSuccess) return ly->cuda_fail(e, "key rotation join");
        }
        // attention launches on the second partition may claim only ready ranges
        const int all_ranges = aa.n_ranges;
        aa.grid = P.sm_attn;  // one attention CTA per SM of the partition
        aa.n_ranges = 1;
        e = timed(ly, PH_ATTN, P.s_attn, [&] { return kvm::launch_attn(aa, bf16, P.s_attn); });
        if (e != cudaSuccess) return ly->cuda_fail(e, "attention launch");
        ly->kernels += 1;
        e = timed(ly, PH_FOLD, P.s_fold, [&] {
            for (int sg = 0; sg < segs; ++sg) {
                fa.e_begin = (int)bnd(sg);
                fa.e_end = (int)bnd(sg + 1);
                cudaError_t r = kvm::launch_fold(fa, bf16, P.s_fold);
                if (r == cudaSuccess) r = cudaEventRecord(P.ev_seg[sg], P.s_fold);
                if (r != cudaSuccess) return r;
                ly->kernels += 1;
                if (L.logs && sg + 1 < segs) {
                    // the segment's snapshots, from its row log, on the attention's SMs (the
                    // last segment's run on every SM, before the last attention launch)
                    rb.e_begin = fa.e_begin;
                    rb.e_end = fa.e_end;
                    r = cudaStreamWaitEvent(P.s_attn, P.ev_seg[sg], 0);
                    if (r == cudaSuccess) r = timed(ly, PH_OTHER, P.s_attn, [&] { return kvm::launch_snap_rebuild(rb, P.s_attn); });
                    if (r == cudaSuccess) r = cudaEventRecord(P.ev_rebuilt, P.s_attn);
                    if (r != cudaSuccess) return r;
                    ly->kernels += 1;
                }
                if (sg + 1 < segs) {
                    r = cudaStreamWaitEvent(P.s_attn, P.ev_seg[sg], 0);
                    aa.n_ranges = sg + 2;
                    if (r == cudaSuccess) r = timed(ly, PH_ATTN, P.s_attn, [&] { return kvm::launch_attn(aa, bf16, P.s_attn); });
                    if (r != cudaSuccess) return r;
                    ly->kernels += 1;
                }
            }
            return cudaSuccess;
        });
        if (e != cudaSuccess) return ly->cuda_fail(e, "overlapped fold / attention launch");
        // what is left of the attention on every SM, once the chain is done (and, with
        // the row log, once the last snapshots are rebuilt)
        e = cudaStreamWaitEvent(s, P.ev_seg[segs - 1], 0);
        if (e == cudaSuccess && L.logs) {
            rb.e_begin = (int)bnd(segs - 1);
            rb.e_end = (int)E;
            // it reads the previous segment's last snapshot, rebuilt on the attention's SMs
            if (segs > 1) e = cudaStreamWaitEvent(s, P.ev_rebuilt, 0);
            if (e == cudaSuccess) e = timed(ly, PH_OTHER, s, [&] { return kvm::launch_snap_rebuild(rb, s); });
            if (e == cudaSuccess) ly->kernels += 1;
        }
        aa.n_ranges = all_ranges;
        aa.grid = P.sm_all;
        if (e == cudaSuccess) e = timed(ly, PH_ATTN, s, [&] { return kvm::launch_attn(aa, bf16, s); });
        if (e != cudaSuccess) return ly->cuda_fail(e, "attention launch");
        ly->kernels += 1;
        e = cudaEventRecord(P.ev_attn, P.s_attn);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, P.ev_attn, 0);
        if (e != cudaSuccess) return ly->cuda_fail(e, "overlap join");
    } else {
        if (E > 0) {
            e = timed(ly, PH_FOLD, s, [&] { return kvm::launch_fold(fa, bf16, s); });
            if (e != cudaSuccess) return ly->cuda_fail(e, "fold chain launch");
            ly->kernels += 1;
            if (L.logs) {
                rb.e_begin = 0;
                rb.e_end = (int)E;
                e = timed(ly, PH_OTHER, s, [&] { return kvm::launch_snap_rebuild(rb, s); });
                if (e != cudaSuccess) return ly->cuda_fail(e, "snapshot rebuild launch");
                ly->kernels += 1;
            }
        }
        if (pre_rotate) {
            ka.grid = 8 * ly->nsm;
            e = timed(ly, PH_OTHER, s, [&] { return kvm::launch_rope_keys(ka, s); });
            if (e != cudaSuccess) return ly->cuda_fail(e, "key rotation launch");
            ly->kernels += 1;
        }
        if (n_tokens > 0) {
            e = timed(ly, PH_ATTN, s, [&] { return kvm::launch_attn(aa, bf16, s); });
            if (e != cudaSuccess) return ly->cuda_fail(e, "attention launch");
            ly->kernels += 1;
        }
    }
    if (ring_work && !pre_rotate) {
        e = timed(ly, PH_OTHER, s, [&] { return kvm::launch_ring_fill(ra, bf16, s); });
        if (e != cudaSuccess) return ly->cuda_fail(e, "ring fill launch");
        ly->kernels += 1;
    }
    ly->n_slots = E > 0 ? ly->sched[E - 1].n_after : 0;
    ly->n_overflow = E * c.chunk;
    ly->pos = n_tokens;
    ly->lse_valid = aa.lse != nullptr;
    return KVM_OK;
}

kvm_status kvm_decode_step(kvm_layer* ly, const void* q, const void* k, const void* v, const float* gate,
                           void* out, void* cuda_stream) {
    NvtxRange nvtx_range("kvm_decode_step");
    if (!ly) { g_err = "layer is NULL"; return KVM_ERR_INVALID_ARG; }
    const kvm_config& c = ly->cfg;
    if (!q || !k || !v || !gate || !out)
        return ly->fail(KVM_ERR_INVALID_ARG, "q, k, v, gate and out must be non-NULL");
    const int64_t p = ly->pos;
    if (p >= c.max_tokens) return ly->fail(KVM_ERR_CAPACITY, "position reached max_tokens");
    DeviceGuard g(ly->device);
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    ly->last_stream = s;
    const bool bf16 = c.dtype == KVM_BF16;
    const int BH = c.batch * c.heads;
    const Layout& L = ly->L;
    const int L_ring = c.window + c.chunk;
    const int64_t ch = p / c.chunk, Wc = c.window / c.chunk;
    int64_t n = ly->n_slots, t = ly->n_overflow;
    const bool fold = (p % c.chunk == 0) && ch >= Wc + 1;
    Sched sc{};
    if (fold) {
        const int64_t ev = ch - Wc - 1;
        sc = event_sched(c, ev * c.chunk, n, t);
        if (sc.n_after > c.max_slots) return ly->fail(KVM_ERR_CAPACITY, "growth schedule exceeds max_slots");
        kvm::FoldArgs fa{};
        fa.sum_k = ly->at<float>(L.sum_k);
        fa.sum_v = ly->at<float>(L.sum_v);
        fa.counts = ly->at<int>(L.counts);
        fa.rho = ly->at<float>(L.rho);
        fa.simdir = ly->at<float>(L.simdir);
        fa.view_k = ly->ws + L.view_k;
        fa.view_v = ly->ws + L.view_v;
        fa.M = c.max_slots;
        fa.C = c.chunk;
        fa.S = c.n_sinks;
        fa.r = c.rope_dims;
        fa.ln_eps = c.ln_eps;
        fa.no_vnorm = (c.flags & KVM_FLAG_NO_VALUE_NORM) != 0;
        fa.k_src = ly->ws + L.ring_k;
        fa.v_src = ly->ws + L.ring_v;
        fa.g_src = ly->at<float>(L.ring_g);
        fa.src_row = L_ring;
        fa.src_len = L_ring;
        fa.e_begin = (int)ev;
        fa.e_end = (int)ev + 1;
        fa.sched = nullptr;
        fa.sched0 = sc;
        fa.status = ly->at<int>(L.status);
        fa.BH = BH;
        cudaError_t e = timed(ly, PH_FOLD, s, [&] { return kvm::launch_fold(fa, bf16, s); });
        if (e != cudaSuccess) return ly->cuda_fail(e, "decode fold launch");
        ly->kernels += 1;
        n = sc.n_after;
        t += c.chunk;
    }
    kvm::DecodeArgs da{};
    da.q = q;
    da.k = k;
    da.v = v;
    da.g = gate;
    da.out = out;
    da.ring_k = ly->ws + L.ring_k;
    da.ring_v = ly->ws + L.ring_v;
    da.ring_g = ly->at<float>(L.ring_g);
    da.ring_kr = ly->ws + L.ring_kr;
    da.view_k = ly->ws + L.view_k;
    da.view_v = ly->ws + L.view_v;
    da.M = c.max_slots;
    da.n_slots = (int)n;
    da.C = c.chunk;
    da.W = c.window;
    da.pos = p;
    da.rope = ly->at<float2>(L.rope);
    da.r = c.rope_dims;
    da.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
    da.BH = BH;
    da.status = ly->at<int>(L.status);
    cudaError_t e = timed(ly, PH_DECODE, s, [&] { return kvm::launch_decode(da, bf16, s); });
    if (e != cudaSuccess) return ly->cuda_fail(e, "decode launch");
    ly->kernels += 1;
    ly->n_slots = n;
    ly->n_overflow = t;
    ly->pos = p + 1;
    ly->lse_valid = false;
    return KVM_OK;
}

static kvm_status copy_state(kvm_layer* ly, kvm_state_bufs* ext, bool to_ext, cudaStream_t s) {
    const kvm_config& c = ly->cfg;
    const Layout& L = ly->L;
    const size_t BH = (size_t)c.batch * c.heads, M = c.max_slots;
    const size_t es = c.dtype == KVM_BF16 ? 2 : 4;
    const size_t ring = (size_t)c.window + c.chunk;
    struct Item { void* ext; size_t off; size_t bytes; } items[] = {
        {ext->sum_k, L.sum_k, BH * M * D * 4}, {ext->sum_v, L.sum_v, BH * M * D * 4},
        {ext->counts, L.counts, BH * M * 4},   {ext->rho, L.rho, BH * M * 4},
        {ext->ring_k, L.ring_k, BH * ring * D * es}, {ext->ring_v, L.ring_v, BH * ring * D * es},
        {ext->ring_g, L.ring_g, BH * ring * 4},
    };
    for (auto& it : items) {
        if (!it.ext) return ly->fail(KVM_ERR_INVALID_ARG, "state buffer pointer is NULL");
    }
    for (auto& it : items) {
        cudaError_t e = to_ext ? cudaMemcpyAsync(it.ext, ly->ws + it.off, it.bytes, cudaMemcpyDeviceToDevice, s)
                               : cudaMemcpyAsync(ly->ws + it.off, it.ext, it.bytes, cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return ly->cuda_fail(e, "state copy");
    }
    return KVM_OK;
}

kvm_status kvm_state_export(const kvm_layer* cly, kvm_state_bufs* dst, void* cuda_stream) {
    NvtxRange nvtx_range("kvm_state_export");
    kvm_layer* ly = const_cast<kvm_layer*>(cly);
    if (!ly) { g_err = "layer is NULL"; return KVM_ERR_INVALID_ARG; }
    if (!dst) return ly->fail(KVM_ERR_INVALID_ARG, "dst is NULL");
    DeviceGuard g(ly->device);
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    ly->last_stream = s;
    kvm_status st = copy_state(ly, dst, true, s);
    if (st != KVM_OK) return st;
    dst->n_slots = ly->n_slots;
    dst->n_overflow = ly->n_overflow;
    dst->pos = ly->pos;
    return KVM_OK;
}

kvm_status kvm_state_import(kvm_layer* ly, const kvm_state_bufs* src, void* cuda_stream) {
    NvtxRange nvtx_range("kvm_state_import");
    if (!ly) { g_err = "layer is NULL"; return KVM_ERR_INVALID_ARG; }
    if (!src) return ly->fail(KVM_ERR_INVALID_ARG, "src is NULL");
    const kvm_config& c = ly->cfg;
    if (src->n_slots < 0 || src->n_slots > c.max_slots) return ly->fail(KVM_ERR_INVALID_ARG, "n_slots out of range");
    if (src->pos < 0 || src->pos > c.max_tokens) return ly->fail(KVM_ERR_INVALID_ARG, "pos out of range");
    if (src->n_overflow < 0 || src->n_overflow > src->pos) return ly->fail(KVM_ERR_INVALID_ARG, "n_overflow out of range");
    DeviceGuard g(ly->device);
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    ly->last_stream = s;
    kvm_state_bufs tmp = *src;
    kvm_status st = copy_state(ly, &tmp, false, s);
    if (st != KVM_OK) return st;
    kvm::RenormArgs ra{};
    const Layout& L = ly->L;
    ra.sum_k = ly->at<float>(L.sum_k);
    ra.sum_v = ly->at<float>(L.sum_v);
    ra.counts = ly->at<int>(L.counts);
    ra.rho = ly->at<float>(L.rho);
    ra.simdir = ly->at<float>(L.simdir);
    ra.view_k = ly->ws + L.view_k;
    ra.view_v = ly->ws + L.view_v;
    ra.M = c.max_slots;
    ra.n = (int)src->n_slots;
    ra.r = c.rope_dims;
    ra.ln_eps = c.ln_eps;
    ra.no_vnorm = (c.flags & KVM_FLAG_NO_VALUE_NORM) != 0;
    ra.BH = c.batch * c.heads;
    ra.status = ly->at<int>(L.status);
    cudaError_t e = timed(ly, PH_OTHER, s, [&] { return kvm::launch_renorm(ra, c.dtype == KVM_BF16, s); });
    if (e != cudaSuccess) return ly->cuda_fail(e, "renormalise launch");
    if (ra.n > 0) ly->kernels += 1;
    // rotated copy of the imported window: tokens at positions [pos - (W + C), pos)
    const int64_t Lr = (int64_t)c.window + c.chunk;
    kvm::RingFillArgs rf{};
    rf.ring_k = ly->ws + L.ring_k;
    rf.ring_v = ly->ws + L.ring_v;
    rf.ring_g = ly->at<float>(L.ring_g);
    rf.ring_kr = ly->ws + L.ring_kr;
    rf.rope = ly->at<float2>(L.rope);
    rf.r = c.rope_dims;
    rf.N = src->pos;
    rf.first = src->pos > Lr ? src->pos - Lr : 0;
    rf.L = (int)Lr;
    rf.BH = c.batch * c.heads;
    rf.rotate_only = 1;
    e = timed(ly, PH_OTHER, s, [&] { return kvm::launch_ring_fill(rf, c.dtype == KVM_BF16, s); });
    if (e != cudaSuccess) return ly->cuda_fail(e, "ring rotation launch");
    if (rf.N > rf.first) ly->kernels += 1;
    ly->n_slots = src->n_slots;
    ly->n_overflow = src->n_overflow;
    ly->pos = src->pos;
    ly->lse_valid = false;
    return KVM_OK;
}

kvm_status kvm_layer_sync(kvm_layer* ly) {
    if (!ly) { g_err = "layer is NULL"; return KVM_ERR_INVALID_ARG; }
    DeviceGuard g(ly->device);
    cudaError_t e = cudaStreamSynchronize(ly->last_stream);
    if (e != cudaSuccess) return ly->cuda_fail(e, "stream synchronise");
    int status = 0;
    e = cudaMemcpy(&status, ly->ws + ly->L.status, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return ly->cuda_fail(e, "status read");
    if (status) {
        cudaMemset(ly->ws + ly->L.status, 0, sizeof(int));
        if (status & kvm::STATUS_TIMEOUT) return ly->fail(KVM_ERR_TIMEOUT, "a bounded device-side wait expired");
        return ly->fail(KVM_ERR_DEVICE, "a device-side consistency check failed");
    }
    return KVM_OK;
}

kvm_status kvm_layer_set_timing(kvm_layer* ly, int enable) {
    if (!ly) { g_err = "layer is NULL"; return KVM_ERR_INVALID_ARG; }
    ly->timing = enable != 0;
    ly->used = 0;
    ly->kernels = 0;
    for (int i = 0; i < 5; ++i) {
        ly->acc_ms[i] = 0.0;
        ly->acc_n[i] = 0;
    }
    return KVM_OK;
}

kvm_status kvm_layer_get_timing(kvm_layer* ly, kvm_timing* out) {
    if (!ly) { g_err = "layer is NULL"; return KVM_ERR_INVALID_ARG; }
    if (!out) return ly->fail(KVM_ERR_INVALID_ARG, "out is NULL");
    DeviceGuard g(ly->device);
    for (size_t i = 0; i < ly->used; ++i) {
        auto& t = ly->pool[i];
        cudaError_t e = cudaEventSynchronize(t.b);
        float ms = 0.0f;
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, t.a, t.b);
        if (e != cudaSuccess) return ly->cuda_fail(e, "timing events");
        ly->acc_ms[t.phase] += ms;
        ly->acc_n[t.phase] += 1;
    }
    ly->used = 0;
    out->fold_ms = ly->acc_ms[PH_FOLD];
    out->attn_ms = ly->acc_ms[PH_ATTN];
    out->decode_ms = ly->acc_ms[PH_DECODE];
    out->other_ms = ly->acc_ms[PH_OTHER];
    out->fold_launches = ly->acc_n[PH_FOLD];
    out->attn_launches = ly->acc_n[PH_ATTN];
    out->decode_launches = ly->acc_n[PH_DECODE];
    out->other_launches = ly->acc_n[PH_OTHER];
    out->kernels = ly->kernels;
    out->proj_ms = ly->acc_ms[PH_PROJ];
    out->proj_launches = ly->acc_n[PH_PROJ];
    return KVM_OK;
}

namespace {
// offsets of q, k, v, o and gate inside the forward scratch
struct FwdScratch {
    size_t q, k, v, o, gate, total;
};
FwdScratch fwd_scratch_of(const kvm_config& c, int64_t n_tokens) {
    FwdScratch f;
    const size_t rows = (size_t)c.batch * c.heads * (size_t)n_tokens;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = kvm::host::align_up(o + bytes); return at; };
    f.q = take(rows * D * 2);
    f.k = take(rows * D * 2);
    f.v = take(rows * D * 2);
    f.o = take(rows * D * 2);
    f.gate = take(rows * 4);
    f.total = o;
    return f;
}
}  // namespace

size_t kvm_forward_scratch_bytes(const kvm_config* cfg, int32_t d_model, int64_t n_tokens) {
    std::string why;
    if (!validate(cfg, why)) { g_err = why; return 0; }
    if (cfg->dtype != KVM_BF16 || d_model < 64 || d_model % 64 || n_tokens < 1 || n_tokens > cfg->max_tokens) {
        g_err = "kvm_forward_scratch_bytes: bf16 layer, d_model a positive multiple of 64, 1 <= n_tokens <= max_tokens";
        return 0;
    }
    return fwd_scratch_of(*cfg, n_tokens).total;
}

kvm_status kvm_layer_forward(kvm_layer* ly, int32_t d_model, const void* x, const void* w_in, const void* w_out,
                             int64_t n_tokens, void* y, void* scratch, size_t scratch_bytes, void* cuda_stream) {
    NvtxRange nvtx_range("kvm_layer_forward");
    if (!ly) { g_err = "layer is NULL"; return KVM_ERR_INVALID_ARG; }
    const kvm_config& c = ly->cfg;
    if (c.dtype != KVM_BF16) return ly->fail(KVM_ERR_UNSUPPORTED, "kvm_layer_forward needs a bf16 layer");
    if (d_model < 64 || d_model % 64) return ly->fail(KVM_ERR_INVALID_ARG, "d_model must be a positive multiple of 64");
    if (n_tokens < 1 || n_tokens > c.max_tokens) return ly->fail(KVM_ERR_INVALID_ARG, "n_tokens must be in [1, max_tokens]");
    if (!x || !w_in || !w_out || !y || !scratch)
        return ly->fail(KVM_ERR_INVALID_ARG, "x, w_in, w_out, y and scratch must be non-NULL");
    for (const void* p : {x, w_in, w_out, (const void*)y})
        if (reinterpret_cast<uintptr_t>(p) % 16) return ly->fail(KVM_ERR_INVALID_ARG, "x, w_in, w_out and y must be 16-byte aligned");
    const FwdScratch F = fwd_scratch_of(c, n_tokens);
    if (reinterpret_cast<uintptr_t>(scratch) % ALIGN || scratch_bytes < F.total)
        return ly->fail(KVM_ERR_WORKSPACE, "scratch missing, misaligned or smaller than kvm_forward_scratch_bytes");
    DeviceGuard g(ly->device);
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    ly->last_stream = s;
    char* sc = static_cast<char*>(scratch);
    const int H = c.heads;
    kvm::GemmSpec in{};
    in.a = x;
    in.w = w_in;
    in.B = c.batch;
    in.N = n_tokens;
    in.H = H;
    in.K = d_model;
    in.Nout = 3 * H * D + H;
    in.a_heads = 0;
    in.epi = 0;
    in.q = sc + F.q;
    in.k = sc + F.k;
    in.v = sc + F.v;
    in.gate = reinterpret_cast<float*>(sc + F.gate);
    in.status = ly->at<int>(ly->L.status);
    cudaError_t e = timed(ly, PH_PROJ, s, [&] { return kvm::launch_gemm_tc(in, s); });
    if (e != cudaSuccess) return ly->cuda_fail(e, "input projection launch");
    ly->kernels += 1;
    kvm_status st = kvm_prefill(ly, sc + F.q, sc + F.k, sc + F.v, reinterpret_cast<const float*>(sc + F.gate),
                                n_tokens, sc + F.o, cuda_stream, nullptr);
    if (st != KVM_OK) return st;
    kvm::GemmSpec outp{};
    outp.a = sc + F.o;
    outp.w = w_out;
    outp.B = c.batch;
    outp.N = n_tokens;
    outp.H = H;
    outp.K = H * D;
    outp.Nout = d_model;
    outp.a_heads = 1;
    outp.epi = 1;
    outp.y = y;
    outp.status = ly->at<int>(ly->L.status);
    e = timed(ly, PH_PROJ, s, [&] { return kvm::launch_gemm_tc(outp, s); });
    if (e != cudaSuccess) return ly->cuda_fail(e, "output projection launch");
    ly->kernels += 1;
    return KVM_OK;
}

namespace {
struct BwdScratch {
    size_t qr, kr, lse, dd, dks, dvs, drho, mem, moff, total;
};
BwdScratch bwd_scratch_of(const kvm_config& c, int64_t n_tokens) {
    BwdScratch b;
    const size_t BH = (size_t)c.batch * c.heads, M = c.max_slots;
    const size_t rows = BH * (size_t)n_tokens, es = c.dtype == KVM_BF16 ? 2 : 4;
    const size_t E = (size_t)kvm::host::n_events_for(c, n_tokens);
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = kvm::host::align_up(o + bytes); return at; };
    b.qr = take(rows * D * es);
    b.kr = take(rows * D * es);
    b.lse = take(rows * 4);
    b.dd = take(rows * 4);
    b.dks = take(BH * E * M * D * 4);
    b.dvs = take(BH * E * M * D * 4);
    b.drho = take(BH * E * M * 4);
    b.mem = take(BH * E * (size_t)c.chunk * 4);
    b.moff = take(BH * (M + 1) * 4);
    b.total = o;
    return b;
}
}  // namespace

size_t kvm_backward_scratch_bytes(const kvm_config* cfg, int64_t n_tokens) {
    std::string why;
    if (!validate(cfg, why)) { g_err = why; return 0; }
    if (n_tokens < 0 || n_tokens > cfg->max_tokens) { g_err = "n_tokens must be in [0, max_tokens]"; return 0; }
    return bwd_scratch_of(*cfg, n_tokens).total;
}

kvm_status kvm_prefill_backward(kvm_layer* ly, const void* q, const void* k, const void* v, const float* gate,
                                const void* out, const void* dout, const kvm_debug* rec, int64_t n_tokens,
                                float* dq, float* dk, float* dv, float* dgate, void* scratch,
                                size_t scratch_bytes, void* cuda_stream) {
    NvtxRange nvtx_range("kvm_prefill_backward");
    if (!ly) { g_err = "layer is NULL"; return KVM_ERR_INVALID_ARG; }
    const kvm_config& c = ly->cfg;
    if (!q || !k || !v || !gate || !out || !dout || !dq || !dk || !dv || !dgate || !scratch)
        return ly->fail(KVM_ERR_INVALID_ARG, "q, k, v, gate, out, dout, dq, dk, dv, dgate and scratch must be non-NULL");
    if (c.chunk > kvm::MAX_BW_C) return ly->fail(KVM_ERR_UNSUPPORTED, "the backward supports chunks of at most 256 tokens");
    if (c.rope_dims % 4) return ly->fail(KVM_ERR_UNSUPPORTED, "the backward needs rope_dims a multiple of 4");
    if (n_tokens < 0 || n_tokens > c.max_tokens) return ly->fail(KVM_ERR_INVALID_ARG, "n_tokens must be in [0, max_tokens]");
    if (n_tokens >= (int64_t(1) << 29)) return ly->fail(KVM_ERR_UNSUPPORTED, "the backward supports fewer than 2^29 tokens");
    const int64_t E = kvm::host::n_events_for(c, n_tokens);
    if (ly->pos != n_tokens || ly->n_overflow != E * c.chunk)
        return ly->fail(KVM_ERR_INVALID_ARG, "the layer's last prefill was not of n_tokens tokens");
    if (E > 0 && (!rec || !rec->assign || !rec->kind || rec->max_events < E))
        return ly->fail(KVM_ERR_INVALID_ARG, "the forward's record (assign and kind of every fold event) is needed");
    const BwdScratch B = bwd_scratch_of(c, n_tokens);
    if (reinterpret_cast<uintptr_t>(scratch) % ALIGN || scratch_bytes < B.total)
        return ly->fail(KVM_ERR_WORKSPACE, "scratch missing, misaligned or smaller than kvm_backward_scratch_bytes");
    DeviceGuard g(ly->device);
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    ly->last_stream = s;
    const Layout& L = ly->L;
    char* sc = static_cast<char*>(scratch);
    kvm::BackwardArgs a{};
    a.q = q;
    a.k = k;
    a.v = v;
    a.g = gate;
    a.out = out;
    a.dout = dout;
    a.assign = rec ? rec->assign : nullptr;
    a.kind = rec ? rec->kind : nullptr;
    a.rec_events = rec ? (int)rec->max_events : 0;
    a.snap_k = ly->ws + L.snap_k;
    a.snap_v = ly->ws + L.snap_v;
    a.snap_events = (int)ly->E_max;
    a.sched = ly->at<kvm::Sched>(L.sched);
    a.rope = ly->at<float2>(L.rope);
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.dg = dgate;
    a.qr = sc + B.qr;
    a.kr = sc + B.kr;
    a.lse = reinterpret_cast<float*>(sc + B.lse);
    a.dd = reinterpret_cast<float*>(sc + B.dd);
    a.lse_fwd = ly->lse_valid ? ly->at<float>(L.lse) : nullptr;
    a.dks = reinterpret_cast<float*>(sc + B.dks);
    a.dvs = reinterpret_cast<float*>(sc + B.dvs);
    a.drho = reinterpret_cast<float*>(sc + B.drho);
    a.mem = reinterpret_cast<int*>(sc + B.mem);
    a.moff = reinterpret_cast<int*>(sc + B.moff);
    a.N = n_tokens;
    a.BH = c.batch * c.heads;
    a.C = c.chunk;
    a.W = c.window;
    a.M = c.max_slots;
    a.r = c.rope_dims;
    a.E = (int)E;
    a.ln_eps = c.ln_eps;
    a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)D));
    a.inv_sqrt_d = (float)(1.0 / std::sqrt((double)D));
    a.no_vnorm = (c.flags & KVM_FLAG_NO_VALUE_NORM) ? 1 : 0;
    a.status = ly->at<int>(L.status);
    cudaError_t e = timed(ly, PH_OTHER, s, [&] { return kvm::launch_backward(a, c.dtype == KVM_BF16, s); });
    if (e != cudaSuccess) return ly->cuda_fail(e, "backward launch");
    // rotation; the tiled products (+ the rotation back of dk) or the four row kernels;
    // the member lists and the slot sweep
    const bool tiled = c.chunk % 64 == 0;
    ly->kernels += 1 + (tiled ? 1 + (c.rope_dims > 0) : 3 + (a.E > 0)) + (a.E > 0 ? 2 : 0);
    return KVM_OK;
}

kvm_status kvm_layer_set_overlap(kvm_layer* ly, int32_t segments) {
    if (!ly) { g_err = "layer is NULL"; return KVM_ERR_INVALID_ARG; }
    ly->overlap_segs = segments < 0 ? -1 : segments;
    return KVM_OK;
}

kvm_status kvm_layer_get_overlap(const kvm_layer* ly, int32_t* last_segments) {
    if (!ly) { g_err = "layer is NULL"; return KVM_ERR_INVALID_ARG; }
    if (!last_segments) return const_cast<kvm_layer*>(ly)->fail(KVM_ERR_INVALID_ARG, "last_segments is NULL");
    *last_segments = ly->last_segs;
    return KVM_OK;
}


const char* kvm_last_error(const kvm_layer* ly) { return ly ? ly->err.c_str() : g_err.c_str(); }

void kvm_layer_destroy(kvm_layer* ly) { delete ly; }

}  // extern "C"
