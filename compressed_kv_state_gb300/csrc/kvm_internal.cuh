// Internal declarations shared by the translation units of libkvm.so.
// Device code for sm_103a; head_dim is fixed at 64 throughout the library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kvm {

constexpr int D = 64;  // head_dim supported by every kernel

// Device status word bits (latched, read and cleared by kvm_layer_sync).
enum : int { STATUS_TIMEOUT = 1, STATUS_DEVICE = 2 };

// Device-side checks of the KVM_DEBUG build (-DKVM_DEBUG): a failed check latches
// STATUS_DEVICE in the layer's status word (kvm_layer_sync then reports
// KVM_ERR_DEVICE) and the caller skips the access it guards.  In normal builds the
// check is compiled out and the access is unconditional.
#ifdef KVM_DEBUG
__device__ __forceinline__ bool kvm_check(bool ok, int* status) {
    if (!ok && status) atomicOr(status, STATUS_DEVICE);
    return ok;
}
#else
__device__ __forceinline__ bool kvm_check(bool, int*) { return true; }
#endif

// Dims kept per row of the state's read-key view: the non-rotary dims [r, D), rounded
// up to a multiple of 8 (16 bytes of bf16) and at least 8; the row holds dims
// [D - view_k_dims(r), D) of the read key.
__host__ __device__ constexpr int view_k_dims(int r) {
    return ((D - r + 7) / 8) * 8 < 8 ? 8 : ((D - r + 7) / 8) * 8;
}

// Per-event schedule entry, computed on the host in double precision (the
// schedule depends only on counts of tokens, never on data).
struct Sched {
    int n_before;  // slots before the event
    int n0;        // slots after this event's sink founding
    int a;         // slots appended by this event
    int n_after;   // slots after the event
};

// ---------------------------------------------------------------- scalars
template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// ------------------------------------------------------------ fold chain
// State of every (b,h) row lives in the workspace:
//   sum_k, sum_v [BH, M, D] fp32; counts [BH, M] int32; rho [BH, M] fp32;
//   simdir [BH, M, D] fp32 = unit(sum_k - mean(sum_k)), the direction the
//   winner-take-all cosine compares against (cosine against LayerNorm(x) is
//   cosine against x - mean(x));
//   view_k [BH, M, view_k_dims(r)] and view_v [BH, M, D] in the I/O dtype = the
//   just-in-time read view.  The read key is zero on the rotary dims [0, r), so
//   view_k stores only its last view_k_dims(r) dims (rounded up to whole 16-byte
//   pieces of bf16); the per-event snapshots keep full rows.
struct FoldArgs {
    float* sum_k;
    float* sum_v;
    int* counts;
    float* rho;
    float* simdir;
    void* view_k;
    void* view_v;
    int M, C, S, r;
    float ln_eps;
    int no_vnorm;  // ablation: read value = sum_v / count instead of rho * unit(sum_v)
    // tokens: row bh, token i of event e sits at src + bh*src_row + ((e*C) % src_len + i)
    const void* k_src;
    const void* v_src;
    const float* g_src;
    int64_t src_row;  // tokens per (b,h) row of the source arrays
    int64_t src_len;  // modulus of the token offset (ring length, or a huge value)
    int e_begin, e_end;
    const Sched* sched;  // device table indexed by event, or nullptr to use sched0
    Sched sched0;
    // per-event snapshots of the read view for the prefill's attention
    void* snap_k;
    void* snap_v;
    int snap_events;  // events per (b,h) row in the snapshot arrays
    // streamed-state chain only: instead of copying every row to the snapshot, each
    // event logs the rows it touched (full bf16 rows [BH, snap_events, C, D], their
    // slots [BH, snap_events, C] and count [BH, snap_events]); launch_snap_rebuild
    // turns the log into the snapshots on other SMs (nullptr: copy as before)
    void* log_k;
    void* log_v;
    int* log_idx;
    int* log_cnt;
    // optional debug record [BH, dbg_events, C]
    int* dbg_assign;
    int* dbg_kind;
    float* dbg_m;
    float* dbg_gap;
    int dbg_events;
    int test_stall;  // wait for a chunk copy that is never issued (bounded-wait test)
    int* status;
    int BH;
    int stage_rows;  // on-chip chain: rows per TMA box of the state sums (set by its launcher)
};

// ------------------------------------------------------------- attention
struct AttnArgs {
    const void* q;
    const void* k;
    const void* v;
    void* out;
    int64_t N;          // tokens per (b,h) row
    int C, W;
    const void* snap_k; // [BH, snap_events, M, D]
    const void* snap_v;
    int snap_events, M;
    const Sched* sched; // events' slot counts (n_after)
    const float2* rope; // [max_tokens, r/2] (cos, sin)
    int r;
    float scale_log2;   // log2(e) / sqrt(D)
    int BH;
    int* status;
    // Tensor-core path only.  Tiles (128 queries of one row) are numbered
    // query-tile-major and split into ranges r = [range_end[r-1], range_end[r])
    // (range_end[-1] = 0).  tile_ctr != nullptr: CTAs claim tiles of ranges
    // 0 .. n_ranges-1 in order, tile range_end[r-1] + atomicAdd(&tile_ctr[r], 1),
    // so launches on several streams share one numbering and every tile is
    // taken once (a counter overshoots only once its range is exhausted).
    // nullptr: every tile, statically strided over the CTAs.
    static constexpr int MAX_RANGES = 24;
    int* tile_ctr;
    int n_ranges;
    int range_end[MAX_RANGES];
    int grid;           // CTAs to launch; 0 = two per SM of the device
    // Tensor-core path: keys already rotated at their own positions (launch_rope_keys),
    // read instead of k for the window; nullptr = rotate window keys in the kernel.
    const void* k_rot;
    // Tensor-core path: queries already rotated at their own positions (the same pass),
    // loaded instead of q; nullptr = each tile rotates its queries in the kernel.
    const void* q_rot;
    // k_rot / q_rot hold only the r rotated dims of each row (RopeKeysArgs::compact)
    int rot_compact;
    // Tensor-core path, optional: fp32 [BH, N] log2-sum-exp of every query's scaled
    // scores (max + log2 of the sum of 2^(s * scale_log2 - max)), for the backward.
    float* lse;
};

// Keys rotated once at their own positions (rotate-half RoPE on dims [0, r)),
// so that the attention need not rotate every window key for every tile that
// sees it.  bf16 [BH, N, D] in and out.
struct RopeKeysArgs {
    const void* k;
    void* k_rot;
    const void* q;   // optional (nullptr: none): queries rotated into q_rot in the same pass
    void* q_rot;
    const float2* rope;  // [max_tokens, r/2] (cos, sin)
    int r;
    int64_t N;
    int BH;
    int grid;            // CTAs to launch (a multiple of the SM count of the launch's partition)
    // compact rows (r == 32): k_rot / q_rot hold only the r rotated dims of each row
    // ([BH, N, r]); the dims past r are read from k / q themselves
    int compact;
    // optional window ring fill in the same pass (ring_k == nullptr: none): tokens
    // [first, N) enter the ring at row position mod L with their unrotated key,
    // value, gate and the rotated key (the same values as ring_fill_kernel writes)
    const void* v;
    const float* g;
    void* ring_k;
    void* ring_v;
    float* ring_g;
    void* ring_kr;
    int64_t first;
    int L;
};

// Snapshots of the read view from the streamed chain's per-event row log: snapshot e
// = snapshot e - 1 (rows < n_after(e)) with the rows event e touched replaced by
// their logged values.  Events [e_begin, e_end) of every row, in order; the
// snapshot of e_begin - 1 must be complete (an earlier call).  bf16.
struct SnapRebuildArgs {
    const void* log_k;
    const void* log_v;
    const int* log_idx;
    const int* log_cnt;
    void* snap_k;
    void* snap_v;
    int snap_events, C, M, BH;
    const Sched* sched;
    int e_begin, e_end;
    int grid;  // CTAs to launch (0: enough for the device)
};
cudaError_t launch_snap_rebuild(const SnapRebuildArgs& a, cudaStream_t s);
bool fold_logs_rows(const FoldArgs& a, bool bf16);  // the streamed chain runs (and logs)

// Backward of a prefill at the forward's fold decisions (kvm_backward.cu).  All
// arrays are device memory; [BH, N, D] rows in the layer's dtype unless noted.
constexpr int MAX_BW_C = 256;  // chunk sizes the backward supports
struct BackwardArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* g;       // [BH, N]
    const void* out;      // the forward's output
    const void* dout;     // gradient of the loss with respect to out
    const int32_t* assign;  // the forward's debug record [BH, rec_events, C]
    const int32_t* kind;
    int rec_events;
    const void* snap_k;   // the forward's read rows after every event [BH, snap_events, M, D]
    const void* snap_v;
    int snap_events;
    const Sched* sched;
    const float2* rope;
    float* dq;            // fp32 [BH, N, D]
    float* dk;
    float* dv;
    float* dg;            // fp32 [BH, N]
    // scratch
    void* qr;             // rotated q and k [BH, N, D]
    void* kr;
    float* lse;           // [BH, N] log2-sum-exp of each query's scores
    float* dd;            // [BH, N] dout . out
    const float* lse_fwd; // [BH, N] the forward's log2-sum-exp per query, or nullptr (recomputed)
    float* dks;           // [BH, E, M, D] read-row gradients, then sum gradients
    float* dvs;
    float* drho;          // [BH, E, M]
    int* mem;             // [BH, E * C] every slot's member tokens in replay order: (t << 2) | kind
    int* moff;            // [BH, M + 1] slot j's members are mem[moff[j] .. moff[j + 1])
    int64_t N;
    int BH, C, W, M, r, E;
    float ln_eps, scale_log2, inv_sqrt_d;
    int no_vnorm;
    int* status;          // a record entry outside [0, M) or of no known kind latches STATUS_DEVICE
};
cudaError_t launch_backward(const BackwardArgs& a, bool bf16, cudaStream_t s);
// The five products on tcgen05 (bf16, chunks a multiple of 128, the forward's
// log2-sum-exp kept); the caller zeroes the gradient accumulators first.
bool bwd_tc5_supported(const BackwardArgs& a, bool bf16);
bool bwd_tc5_owns_read_rows(const BackwardArgs& a);  // it stores (not adds) the read rows' gradients
cudaError_t launch_bwd_tc5(const BackwardArgs& a, cudaStream_t s);

struct DecodeArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    void* out;
    void* ring_k;
    void* ring_v;
    float* ring_g;
    void* ring_kr;  // window keys with RoPE applied at their own positions
    const void* view_k;
    const void* view_v;
    int M, n_slots, C, W;
    int64_t pos;
    const float2* rope;
    int r;
    float scale_log2;
    int BH;
    int* status;
};

struct RingFillArgs {
    const void* k;      // source keys [BH, N, D] (unrotated)
    const void* v;
    const float* g;
    void* ring_k;
    void* ring_v;
    float* ring_g;
    void* ring_kr;      // rotated copy of the ring keys
    const float2* rope;
    int r;
    int64_t N, first;  // copy tokens [first, N) of each row
    int L;             // ring length W + C
    int BH;
    int rotate_only;   // 1: only recompute ring_kr from ring_k for positions [first, N)
};

struct RenormArgs {
    const float* sum_k;
    const float* sum_v;
    const int* counts;
    const float* rho;
    float* simdir;
    void* view_k;
    void* view_v;
    int M, n, r;
    float ln_eps;
    int no_vnorm;  // ablation: read value = sum_v / count
    int BH;
    int* status;   // device status word (device-side checks of the debug build)
};

// Projection GEMM of the whole layer: C = A * W^T, A [rows, K] bf16 (or the
// attention output [B*H, N, 64] read head by head when a_heads), W [Nout, K]
// bf16; epi 0 scatters q/k/v [B,H,N,64] bf16 and sigmoid gates [B,H,N] fp32,
// epi 1 writes y [B, N, Nout] bf16.  K a multiple of 64.
struct GemmSpec {
    const void* a;
    const void* w;
    int B;
    int64_t N;
    int H, K, Nout;
    int a_heads, epi;
    void* q;
    void* k;
    void* v;
    float* gate;
    void* y;
    int* status;
};

// Host launchers (return the launch error).
cudaError_t launch_fold(const FoldArgs& a, bool bf16, cudaStream_t s);
bool fold_tc_supported(const FoldArgs& a, bool bf16);
cudaError_t launch_fold_tc(const FoldArgs& a, cudaStream_t s);
bool fold_big_supported(const FoldArgs& a, bool bf16);
cudaError_t launch_fold_big(const FoldArgs& a, cudaStream_t s);
cudaError_t launch_attn(const AttnArgs& a, bool bf16, cudaStream_t s);
bool attn_tc_supported(const AttnArgs& a, bool bf16);
cudaError_t launch_attn_tc(const AttnArgs& a, int* status, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs& a, bool bf16, cudaStream_t s);
cudaError_t launch_ring_fill(const RingFillArgs& a, bool bf16, cudaStream_t s);
cudaError_t launch_rope_keys(const RopeKeysArgs& a, cudaStream_t s);
cudaError_t launch_gemm_tc(const GemmSpec& g, cudaStream_t s);
cudaError_t launch_renorm(const RenormArgs& a, bool bf16, cudaStream_t s);
// RoPE table [n_pos, r/2] of (cos, sin) of p * theta^(-2i/r), built on the device
// (angles and their cosine and sine in double precision, stored as float): every
// entry point that needs the table builds it with this one kernel, so their
// tables are identical bit for bit.
cudaError_t launch_rope_table(int rope_dims, float rope_theta, int64_t n_pos, float2* out, cudaStream_t s);

}  // namespace kvm
