// Spatial partition of the GPU's SMs for the overlapped prefill: one green
// context holds the SMs the fold chain runs on (one CTA per (b,h) row, each
// holding a whole SM), a second one holds the rest, where the attention of the
// chunks the chain has already folded runs meanwhile.  Both partitions are
// disjoint, so attention CTAs can never take an SM the next fold segment
// needs.  Work launched on ordinary streams may still use every SM.
//
// Driver entry points are resolved at run time through the runtime, so the
// library links no driver library.  No partition is made while a CUDA
// injection library (a profiler) is attached: kernel profilers do not handle
// launches into green contexts, so under one the prefill runs sequentially.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdlib>
#include <mutex>
#include <string>

#include "kvm_host.h"

namespace kvm {
namespace host {

namespace {

struct Driver {
    PFN_cuDeviceGet_v2000 device_get = nullptr;
    PFN_cuDeviceGetDevResource_v12040 get_resource = nullptr;
    PFN_cuDevSmResourceSplitByCount_v12040 split = nullptr;
    PFN_cuDevResourceGenerateDesc_v12040 gen_desc = nullptr;
    PFN_cuGreenCtxCreate_v12040 gctx_create = nullptr;
    PFN_cuGreenCtxDestroy_v12040 gctx_destroy = nullptr;
    PFN_cuGreenCtxStreamCreate_v12050 gstream_create = nullptr;
    PFN_cuCtxFromGreenCtx_v12040 ctx_from_green = nullptr;
    PFN_cuCtxPushCurrent_v4000 push = nullptr;
    PFN_cuCtxPopCurrent_v4000 pop = nullptr;
    PFN_cuStreamDestroy_v4000 stream_destroy = nullptr;
    bool ok = false;
};

template <class F> bool resolve(const char* name, int version, F* fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p) {
        cudaGetLastError();
        return false;
    }
    *fn = reinterpret_cast<F>(p);
    return true;
}

const Driver& driver() {
    static Driver d;
    static std::once_flag once;
    std::call_once(once, [] {
        d.ok = resolve("cuDeviceGet", 2000, &d.device_get) &&
               resolve("cuDeviceGetDevResource", 12040, &d.get_resource) &&
               resolve("cuDevSmResourceSplitByCount", 12040, &d.split) &&
               resolve("cuDevResourceGenerateDesc", 12040, &d.gen_desc) &&
               resolve("cuGreenCtxCreate", 12040, &d.gctx_create) &&
               resolve("cuGreenCtxDestroy", 12040, &d.gctx_destroy) &&
               resolve("cuGreenCtxStreamCreate", 12050, &d.gstream_create) &&
               resolve("cuCtxFromGreenCtx", 12040, &d.ctx_from_green) &&
               resolve("cuCtxPushCurrent", 4000, &d.push) && resolve("cuCtxPopCurrent", 4000, &d.pop) &&
               resolve("cuStreamDestroy", 4000, &d.stream_destroy);
    });
    return d;
}

// Create n events (timing disabled) that belong to green context g.
bool events_in(const Driver& d, CUgreenCtx g, cudaEvent_t* ev, int n) {
    CUcontext c = nullptr;
    if (d.ctx_from_green(&c, g) != CUDA_SUCCESS || d.push(c) != CUDA_SUCCESS) return false;
    bool ok = true;
    for (int i = 0; i < n && ok; ++i) ok = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) == cudaSuccess;
    CUcontext popped = nullptr;
    d.pop(&popped);
    return ok;
}

}  // namespace

bool partition_make(int device, int fold_rows, Partition* p, std::string& why) {
    *p = Partition{};
    const char* inj = std::getenv("CUDA_INJECTION64_PATH");
    if (inj != nullptr && inj[0] != '\0') { why = "a CUDA injection library (profiler) is attached"; return false; }
    const Driver& d = driver();
    if (!d.ok) { why = "green-context driver entry points unavailable"; return false; }
    CUdevice dev;
    CUdevResource all;
    if (d.device_get(&dev, device) != CUDA_SUCCESS ||
        d.get_resource(dev, &all, CU_DEV_RESOURCE_TYPE_SM) != CUDA_SUCCESS) {
        why = "SM resource query failed";
        return false;
    }
    const unsigned total = all.sm.smCount;
    const unsigned gran = all.sm.smCoscheduledAlignment > 0 ? all.sm.smCoscheduledAlignment : 8;
    const unsigned want = ((unsigned)fold_rows + gran - 1) / gran * gran;
    if (want + all.sm.minSmPartitionSize > total) { why = "too few SMs left beside the fold chain"; return false; }
    CUdevResource grp, rem;
    unsigned nb = 1;
    if (d.split(&grp, &nb, &all, &rem, 0, want) != CUDA_SUCCESS || nb != 1 ||
        grp.sm.smCount < (unsigned)fold_rows || rem.sm.smCount == 0) {
        why = "SM split failed";
        return false;
    }
    CUdevResourceDesc d1, d2;
    CUgreenCtx g1 = nullptr, g2 = nullptr;
    if (d.gen_desc(&d1, &grp, 1) != CUDA_SUCCESS || d.gen_desc(&d2, &rem, 1) != CUDA_SUCCESS ||
        d.gctx_create(&g1, d1, dev, CU_GREEN_CTX_DEFAULT_STREAM) != CUDA_SUCCESS) {
        why = "green context creation failed";
        return false;
    }
    if (d.gctx_create(&g2, d2, dev, CU_GREEN_CTX_DEFAULT_STREAM) != CUDA_SUCCESS) {
        d.gctx_destroy(g1);
        why = "green context creation failed";
        return false;
    }
    p->g_fold = g1;
    p->g_attn = g2;
    CUstream s1 = nullptr, s2 = nullptr;
    if (d.gstream_create(&s1, g1, CU_STREAM_NON_BLOCKING, 0) != CUDA_SUCCESS ||
        d.gstream_create(&s2, g2, CU_STREAM_NON_BLOCKING, 0) != CUDA_SUCCESS) {
        if (s1) d.stream_destroy(s1);
        p->s_fold = nullptr;
        partition_free(p);
        why = "green context stream creation failed";
        return false;
    }
    p->s_fold = reinterpret_cast<cudaStream_t>(s1);
    p->s_attn = reinterpret_cast<cudaStream_t>(s2);
    if (!events_in(d, g1, p->ev_seg, Partition::MAX_SEGS) || !events_in(d, g2, &p->ev_attn, 1) ||
        !events_in(d, g2, &p->ev_rebuilt, 1) ||
        cudaEventCreateWithFlags(&p->ev_fork, cudaEventDisableTiming) != cudaSuccess) {
        partition_free(p);
        why = "event creation failed";
        return false;
    }
    p->sm_fold = (int)grp.sm.smCount;
    p->sm_attn = (int)rem.sm.smCount;
    p->sm_all = (int)total;
    p->ok = true;
    return true;
}

void partition_free(Partition* p) {
    const Driver& d = driver();
    if (p->s_fold) cudaStreamSynchronize(p->s_fold);
    if (p->s_attn) cudaStreamSynchronize(p->s_attn);
    for (auto& e : p->ev_seg)
        if (e) cudaEventDestroy(e);
    if (p->ev_attn) cudaEventDestroy(p->ev_attn);
    if (p->ev_rebuilt) cudaEventDestroy(p->ev_rebuilt);
    if (p->ev_fork) cudaEventDestroy(p->ev_fork);
    if (d.ok) {
        if (p->s_fold) d.stream_destroy(reinterpret_cast<CUstream>(p->s_fold));
        if (p->s_attn) d.stream_destroy(reinterpret_cast<CUstream>(p->s_attn));
        if (p->g_fold) d.gctx_destroy(static_cast<CUgreenCtx>(p->g_fold));
        if (p->g_attn) d.gctx_destroy(static_cast<CUgreenCtx>(p->g_attn));
    }
    cudaGetLastError();
    *p = Partition{};
}

}  // namespace host
}  // namespace kvm
