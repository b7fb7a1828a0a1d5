// Host-side helpers of libkvm.so shared between translation units:
// configuration validation, workspace layout and the data-independent
// growth schedule.  Defined in kvm_api.cu.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <string>

#include "../../include/kvm.h"
#include "kvm_internal.cuh"

namespace kvm {
namespace host {

constexpr size_t ALIGN = 256;

// Byte offsets of every array inside a layer's workspace.
struct Layout {
    size_t sum_k, sum_v, counts, rho, simdir, view_k, view_v;
    size_t ring_k, ring_v, ring_g, ring_kr, snap_k, snap_v, rope, sched, status;
    size_t k_rot;  // keys rotated at their own positions (bf16 layers with rope_dims > 0; else empty)
    size_t q_rot;  // queries rotated at their own positions (same condition)
    size_t log_k, log_v, log_idx, log_cnt;  // the streamed chain's row log (empty otherwise)
    bool logs;
    size_t lse;    // log2-sum-exp of every query's scores, written by the tensor-core attention
    bool has_lse;  // (bf16 layers with chunks a multiple of 128; else empty)
    size_t total;
};

extern thread_local std::string g_err;

size_t align_up(size_t x);
int64_t n_events_for(const kvm_config& c, int64_t N);
int64_t capacity(const kvm_config& c, int64_t t);
Sched event_sched(const kvm_config& c, int64_t first_pos, int64_t n, int64_t t);
bool validate(const kvm_config* c, std::string& why);
Layout layout_of(const kvm_config& c);

// Byte offset, inside the status region, of the attention's tile-range counters.
constexpr size_t TILE_CTR_OFF = 128;

// Two disjoint SM partitions (green contexts) with a stream each, for the
// overlapped prefill; defined in kvm_partition.cu.
struct Partition {
    static constexpr int MAX_SEGS = 16;
    bool ok = false;
    int sm_fold = 0, sm_attn = 0, sm_all = 0;
    void* g_fold = nullptr;  // CUgreenCtx
    void* g_attn = nullptr;
    cudaStream_t s_fold = nullptr, s_attn = nullptr;
    cudaEvent_t ev_fork = nullptr;              // primary context
    cudaEvent_t ev_seg[MAX_SEGS] = {};          // fold partition: end of segment k
    cudaEvent_t ev_attn = nullptr;              // attention partition: end of its work
    cudaEvent_t ev_rebuilt = nullptr;           // attention partition: snapshots of a segment rebuilt
};
// fold_rows SMs (rounded up to the split granularity) for the fold chain, the
// rest for attention.  False (with the reason) when the device or driver
// cannot provide both.
bool partition_make(int device, int fold_rows, Partition* p, std::string& why);
void partition_free(Partition* p);

}  // namespace host
}  // namespace kvm
