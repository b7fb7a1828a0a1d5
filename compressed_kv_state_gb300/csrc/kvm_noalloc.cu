// kvm_prefill_noalloc: a one-shot KVM prefill that allocates no memory.
//
// Who needs it: some callers may not allocate device memory themselves -
// for example a plugin running inside an inference server or another host
// framework that owns every byte of device memory through its own pool and
// forbids direct cudaMalloc/cudaFree (a stray allocation would bypass its
// accounting or fragment its pool), or a latency-critical loop where the
// implicit device synchronisation of cudaMalloc/cudaFree would stall the
// pipeline.  Such callers cannot provide the workspace that kvm_layer_create
// needs.  This entry point runs the same fold-chain and attention kernels as
// kvm_prefill, with the workspace placed in the file-scope device array
// below instead of caller memory.
//
// The array holds KVM_NOALLOC_SCRATCH_BYTES bytes on every GPU that loads
// this library and stays reserved until the process exits.  Every call uses
// the same array and it keeps the previous call's contents, so each call
// clears what must start at zero; calls whose GPU work overlaps (other
// streams, other host threads) race on it.
#include <cmath>
#include <mutex>
#include <string>

#include "../../include/kvm.h"
#include "kvm_host.h"
#include "kvm_internal.cuh"

namespace {

constexpr int MAX_DEVICES = 64;
constexpr int MAX_EVENTS = 1024;  // schedule entries passed by kernel parameter (16 KB)

static __device__ __align__(256) unsigned char g_noalloc_scratch[KVM_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void* g_scratch_addr[MAX_DEVICES] = {};

struct SchedUpload {
    int n;
    kvm::Sched s[MAX_EVENTS];
};

__global__ void sched_upload_kernel(const SchedUpload u, kvm::Sched* dst) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < u.n; i += gridDim.x * blockDim.x) dst[i] = u.s[i];
}

// Device address of the static array on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" kvm_status kvm_prefill_noalloc(const kvm_config* cfg_in, const void* q, const void* k,
                                          const void* v, const float* gate, int64_t n_tokens, void* out,
                                          void* cuda_stream) {
    using namespace kvm::host;
    std::string why;
    if (!validate(cfg_in, why)) {
        g_err = why;
        return KVM_ERR_INVALID_ARG;
    }
    if (n_tokens < 0 || n_tokens > cfg_in->max_tokens) {
        g_err = "n_tokens must be in [0, max_tokens]";
        return KVM_ERR_INVALID_ARG;
    }
    if (n_tokens == 0) return KVM_OK;
    // size the scratch for exactly this call
    kvm_config c = *cfg_in;
    c.max_tokens = (int32_t)n_tokens;
    const Layout L = layout_of(c);
    if (L.total > (size_t)KVM_NOALLOC_SCRATCH_BYTES) {
        g_err = "kvm_prefill_noalloc: this call needs " + std::to_string(L.total) +
                " bytes of scratch, more than the static " + std::to_string((size_t)KVM_NOALLOC_SCRATCH_BYTES) +
                " bytes (KVM_NOALLOC_SCRATCH_BYTES); use kvm_layer_create with a caller workspace";
        return KVM_ERR_WORKSPACE;
    }
    if (!q || !k || !v || !gate || !out) {
        g_err = "q, k, v, gate and out must be non-NULL";
        return KVM_ERR_INVALID_ARG;
    }
    // every buffer must be device memory of the current device (the one whose
    // scratch array and stream this call uses); cudaPointerGetAttributes allocates nothing
    {
        int dev = -1;
        cudaError_t de = cudaGetDevice(&dev);
        if (de != cudaSuccess) {
            g_err = std::string("kvm_prefill_noalloc: cudaGetDevice: ") + cudaGetErrorString(de);
            return KVM_ERR_CUDA;
        }
        const void* ptrs[5] = {q, k, v, gate, out};
        const char* names[5] = {"q", "k", "v", "gate", "out"};
        for (int i = 0; i < 5; ++i) {
            cudaPointerAttributes at;
            const cudaError_t pe = cudaPointerGetAttributes(&at, ptrs[i]);
            if (pe != cudaSuccess) cudaGetLastError();
            if (pe != cudaSuccess ||
                (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged) || at.device != dev) {
                g_err = std::string("kvm_prefill_noalloc: ") + names[i] +
                        " is not device memory of the current device " + std::to_string(dev);
                return KVM_ERR_INVALID_ARG;
            }
        }
    }
    const int64_t E = n_events_for(c, n_tokens);
    if (E > MAX_EVENTS) {
        g_err = "kvm_prefill_noalloc: at most 1024 fold events per call";
        return KVM_ERR_WORKSPACE;
    }
    SchedUpload up;
    up.n = (int)E;
    int64_t n = 0, t = 0;
    for (int64_t ev = 0; ev < E; ++ev) {
        up.s[ev] = event_sched(c, ev * c.chunk, n, t);
        n = up.s[ev].n_after;
        t += c.chunk;
    }
    if (E > 0 && n > c.max_slots) {
        g_err = "growth schedule exceeds max_slots for this n_tokens";
        return KVM_ERR_CAPACITY;
    }
    void* base = nullptr;
    cudaError_t e = scratch_address(&base);
    if (e != cudaSuccess) {
        g_err = std::string("kvm_prefill_noalloc: cudaGetSymbolAddress: ") + cudaGetErrorString(e);
        return KVM_ERR_CUDA;
    }
    char* ws = static_cast<char*>(base);
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    const bool bf16 = c.dtype == KVM_BF16;
    const int BH = c.batch * c.heads;

    // what must start at zero: counts, the status word, and the snapshot rows
    // beyond each snapshot's slot count (read and masked by the attention)
    e = cudaMemsetAsync(ws + L.counts, 0, L.rho - L.counts, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(ws + L.status, 0, 16, s);
    if (e == cudaSuccess && L.rope > L.snap_k) e = cudaMemsetAsync(ws + L.snap_k, 0, L.rope - L.snap_k, s);
    if (e == cudaSuccess && E > 0) {
        sched_upload_kernel<<<1, 256, 0, s>>>(up, reinterpret_cast<kvm::Sched*>(ws + L.sched));
        e = cudaGetLastError();
    }
    if (e == cudaSuccess)
        e = kvm::launch_rope_table(c.rope_dims, c.rope_theta, n_tokens, reinterpret_cast<float2*>(ws + L.rope), s);
    if (e == cudaSuccess && E > 0) {
        kvm::FoldArgs fa{};
        fa.sum_k = reinterpret_cast<float*>(ws + L.sum_k);
        fa.sum_v = reinterpret_cast<float*>(ws + L.sum_v);
        fa.counts = reinterpret_cast<int*>(ws + L.counts);
        fa.rho = reinterpret_cast<float*>(ws + L.rho);
        fa.simdir = reinterpret_cast<float*>(ws + L.simdir);
        fa.view_k = ws + L.view_k;
        fa.view_v = ws + L.view_v;
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
        fa.sched = reinterpret_cast<const kvm::Sched*>(ws + L.sched);
        fa.snap_k = ws + L.snap_k;
        fa.snap_v = ws + L.snap_v;
        fa.snap_events = (int)E;
        fa.status = reinterpret_cast<int*>(ws + L.status);
        fa.BH = BH;
        if (L.logs) {
            fa.log_k = ws + L.log_k;
            fa.log_v = ws + L.log_v;
            fa.log_idx = reinterpret_cast<int*>(ws + L.log_idx);
            fa.log_cnt = reinterpret_cast<int*>(ws + L.log_cnt);
        }
        e = kvm::launch_fold(fa, bf16, s);
        if (e == cudaSuccess && L.logs) {
            // the snapshots, from the chain's row log
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
            rb.BH = BH;
            rb.sched = fa.sched;
            rb.e_begin = 0;
            rb.e_end = (int)E;
            e = kvm::launch_snap_rebuild(rb, s);
        }
    }
    kvm::AttnArgs aa{};
    aa.q = q;
    aa.k = k;
    aa.v = v;
    aa.out = out;
    aa.N = n_tokens;
    aa.C = c.chunk;
    aa.W = c.window;
    aa.snap_k = ws + L.snap_k;
    aa.snap_v = ws + L.snap_v;
    aa.snap_events = (int)E;
    aa.M = c.max_slots;
    aa.sched = reinterpret_cast<const kvm::Sched*>(ws + L.sched);
    aa.rope = reinterpret_cast<const float2*>(ws + L.rope);
    aa.r = c.rope_dims;
    aa.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)kvm::D));
    aa.BH = BH;
    aa.status = reinterpret_cast<int*>(ws + L.status);
    // tensor-core attention: keys rotated once, before it
    if (e == cudaSuccess && bf16 && c.rope_dims > 0 && kvm::attn_tc_supported(aa, bf16)) {
        int dev = 0, nsm = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        kvm::RopeKeysArgs ka{};
        ka.k = k;
        ka.k_rot = ws + L.k_rot;
        ka.q = q;
        ka.q_rot = ws + L.q_rot;
        ka.rope = aa.rope;
        ka.r = c.rope_dims;
        ka.N = n_tokens;
        ka.BH = BH;
        ka.grid = 8 * (nsm > 0 ? nsm : 1);
        ka.compact = c.rope_dims == 32;
        e = kvm::launch_rope_keys(ka, s);
        aa.k_rot = ka.k_rot;
        aa.q_rot = ka.q_rot;
        aa.rot_compact = ka.compact;
    }
    if (e == cudaSuccess) e = kvm::launch_attn(aa, bf16, s);
    if (e != cudaSuccess) {
        g_err = std::string("kvm_prefill_noalloc: ") + cudaGetErrorString(e);
        return KVM_ERR_CUDA;
    }
    return KVM_OK;
}
