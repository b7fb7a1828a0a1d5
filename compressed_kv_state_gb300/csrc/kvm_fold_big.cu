// Fold chain on the tensor cores for large states (bf16 I/O, any max_slots up
// to 4096, chunks up to 256 tokens): the case the on-chip chain (state in
// tensor memory, at most 256 slots and 128 tokens) does not cover.
//
// "Key-Value Means" (gist.science technical summary), Core mechanisms 1-3
// and 5 (the growable "KVM sqrt" state of Core mechanism 3 reaches hundreds to
// thousands of slots); lay part "smart merge".  Same rule as the other fold
// chains.  One CTA of 512 threads runs one (b, h) row's events back to back;
// the state stays in the workspace (it fits in L2), and per event:
//   - the winner-take-all directions u_j = unit(sum_k_j - mean) live in the
//     workspace as bf16 hi + lo rows; TMA streams them through shared memory
//     in blocks of NB slots (double-buffered), and the similarity of the
//     chunk's keys to each block is a tcgen05 MMA chain into one of two
//     tensor-memory buffers, so block b + 1 multiplies while block b is
//     scanned (four threads per token, 64 slot columns each, running best /
//     second / argmax in registers);
//   - chunks of up to 256 tokens are two 128-row MMA tiles (NB = 128 then,
//     else NB = 256: each S buffer is 256 tensor-memory columns);
//   - the slots the event touches are compacted (a slot bitmap, prefix counts
//     and per-slot 256-bit token masks); eight lanes per touched slot (eight
//     dims each, four slots per warp at a time) add its tokens in position
//     order, then write the new direction, the read view and the sums back;
//   - the read view of every slot is copied to the event's snapshot.
// The merge is deterministic: no atomics on data (token masks are OR-ed).
#include <cstddef>

#include "kvm_internal.cuh"
#include "tc_primitives.cuh"

namespace kvm {
namespace foldbig {

using namespace tc;

constexpr int NT = 512;       // threads
constexpr int NW = NT / 32;   // warps
constexpr int MAXC = 256;     // tokens per event
constexpr int MAXM = 4096;    // slots
constexpr int ROWB = 128;     // bytes of a 64-dim bf16 row
constexpr int TILE_BYTES = 128 * ROWB;  // 128 token rows

struct Misc {
    // 8-byte barriers first, then the 16-byte-accessed masks (the struct starts
    // 1024-byte aligned)
    unsigned long long bar_k[2], bar_u[2], bar_s[2];
    uint32_t tmem_slot;
    int abort_flag;
    alignas(16) uint32_t tmask[MAXC][MAXC / 32];  // merged tokens of a touched slot
    float g[MAXC], kn[MAXC], m[MAXC];
    float pb[4][MAXC], ps[4][MAXC];  // per-thread partial best / second best
    int pa[4][MAXC];                 // and argmax
    int kind[MAXC], slot[MAXC];
    uint32_t slotbits[MAXM / 32];    // slots the event touches
    int wbase[MAXM / 32 + 4];        // prefix counts of slotbits (compact index of a slot)
    int tslot[MAXC];                 // touched slot of each compact index
    int kfound[MAXC];                // founding token of a touched slot (-1: merges only)
    int wapp[NW];                    // appended tokens per warp (selection order)
};
static_assert(offsetof(Misc, tmask) % 16 == 0, "token masks are read as 16-byte vectors");
#ifdef KVM_PROBE
static __device__ unsigned long long g_probe_big[32];
#endif
constexpr int BODY_BYTES = 192 * 1024;  // U blocks + chunk buffers (either tiling)
constexpr int SMEM_BYTES = BODY_BYTES + (int)sizeof(Misc) + 1024;

__device__ __forceinline__ int swz(int row, int ch) { return row * ROWB + (((ch ^ (row & 7)) & 7) << 4); }
// dims (2l, 2l + 1) of a 128-byte swizzled bf16 row, as a float2
__device__ __forceinline__ float2 row_pair(const uint8_t* base, int row, int l) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(base + swz(row, l >> 2) + ((l & 3) << 2));
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// (b, s, arg) <- best / second best / argmax of two partial results over
// disjoint slot sets (ties go to the lower slot index)
__device__ __forceinline__ void combine(float& b, float& s, int& arg, float b2, float s2, int a2) {
    if (a2 < 0) return;
    if (arg < 0) {
        b = b2;
        s = s2;
        arg = a2;
        return;
    }
    if (b2 > b || (b2 == b && a2 < arg)) {
        s = fmaxf(fmaxf(s, s2), b);
        b = b2;
        arg = a2;
    } else {
        s = fmaxf(fmaxf(s, s2), b2);
    }
}

// Running best / argmax (and, with GAP, second best) over 32 columns of slots
// base .. base + 31 restricted to [lo, hi); slots increase along the scan, so a
// strictly larger value takes the lead and ties keep the lower index.
template <bool GAP>
__device__ __forceinline__ void scan32(const uint32_t (&v)[32], int base, int lo, int hi, float& b, float& s,
                                       int& arg) {
    if (base >= lo && base + 32 <= hi) {
#pragma unroll
        for (int x = 0; x < 32; ++x) {
            const float val = __uint_as_float(v[x]);
            arg = val > b ? base + x : arg;
            if (GAP) s = fmaxf(s, fminf(val, b));
            b = fmaxf(b, val);
        }
    } else if (base + 32 > lo && base < hi) {
#pragma unroll
        for (int x = 0; x < 32; ++x) {
            const int j = base + x;
            const float val = (j >= lo && j < hi) ? __uint_as_float(v[x]) : -INFINITY;
            arg = val > b ? j : arg;
            if (GAP) s = fmaxf(s, fminf(val, b));
            b = fmaxf(b, val);
        }
    }
}

// One warp renormalises slot j from its key sums x (dims 2l, 2l + 1 on lane l):
// writes the direction u = unit(x - mean) as bf16 hi + lo into the workspace row
// (hi at elements [0, 64), lo at [64, 128)) and returns the centred pair and |c|^2.
__device__ __forceinline__ float warp_dir(float2 x, int l, __nv_bfloat16* urow, float2& c, uint32_t& hi_out,
                                         uint32_t& lo_out) {
    const float mean = warp_sum(x.x + x.y) * (1.0f / 64.0f);
    c = make_float2(x.x - mean, x.y - mean);
    const float ss = warp_sum(c.x * c.x + c.y * c.y);
    const float inv = ss > 0.0f ? 1.0f / sqrtf(ss) : 0.0f;
    const float ux = c.x * inv, uy = c.y * inv;
    const uint32_t hi = pack2(ux, uy);
    const float2 hf = unpack2(hi);
    const uint32_t lo = pack2(ux - hf.x, uy - hf.y);
    reinterpret_cast<uint32_t*>(urow)[l] = hi;
    reinterpret_cast<uint32_t*>(urow)[32 + l] = lo;
    hi_out = hi;
    lo_out = lo;
    return ss;
}

template <bool GAP>
__global__ void __launch_bounds__(NT, 1)
    fold_big_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_u, const FoldArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    Misc& X = *reinterpret_cast<Misc*>(sm + BODY_BYTES);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x;
    const int C = a.C, S = a.S, M = a.M;
    const int T = C > 128 ? 2 : 1;       // 128-token MMA tiles per chunk
    const int NB = 256 / T;              // slots per similarity block
    const int UBUF = NB * ROWB * 2;      // one U block: hi rows then lo rows
    const int OFF_K = 2 * UBUF;
    const int CHB = T * TILE_BYTES;      // one chunk buffer (keys or values)
    const int OFF_V = OFF_K + 2 * CHB;

    float* g_sk = a.sum_k + (int64_t)bh * M * D;
    float* g_sv = a.sum_v + (int64_t)bh * M * D;
    int* g_cnt = a.counts + (int64_t)bh * M;
    float* g_rho = a.rho + (int64_t)bh * M;
    __nv_bfloat16* g_u = reinterpret_cast<__nv_bfloat16*>(a.simdir) + (int64_t)bh * M * 128;
    const int DK = view_k_dims(a.r), zc = (D - DK) / 8;  // compact read-key rows: 16-byte pieces zc..7
    __nv_bfloat16* g_vk = reinterpret_cast<__nv_bfloat16*>(a.view_k) + (int64_t)bh * M * DK;
    __nv_bfloat16* g_vv = reinterpret_cast<__nv_bfloat16*>(a.view_v) + (int64_t)bh * M * D;

    const Sched sc_first = a.sched ? a.sched[a.e_begin] : a.sched0;
    int n = sc_first.n_before;
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&X.bar_k[i]), 1);
            mbar_init(smem_u32(&X.bar_u[i]), 1);
            mbar_init(smem_u32(&X.bar_s[i]), 2);  // one commit from each issuer
        }
        X.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(&X.tmem_slot), 512);
    // the directions of the slots the state already holds are in the workspace: written
    // by the events that touched them, or by the state import's renormalisation
    fence_proxy_async_all();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = X.tmem_slot;
    const uint32_t sbase = smem_u32(sm);
    const uint32_t idesc = idesc_bf16(128, 128, 0, 0);
    // two threads in different warps issue a block's similarity MMAs, each half of them
    // (issuing holds the thread about as long as the tensor core takes the MMAs, and the
    // issuing warp scans only after it): thread 0 takes k = 0, thread ISS2 k = 1
    constexpr int ISS2 = 256;
    const bool issuer = tid == 0 || tid == ISS2;
    const int ik = tid == 0 ? 0 : 1;
    const int q = warp & 3, G = warp >> 2;  // TMEM lane quarter, column group
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    // this thread's token row and the 64 slot columns it scans in a block
    const int tok = (T == 1 ? 0 : (G >> 1) * 128) + q * 32 + lane;
    const int colslot = T == 1 ? 64 * G : 64 * (G & 1);
    const int part = T == 1 ? G : (G & 1);
    const int nparts = T == 1 ? 4 : 2;

    // thread 0's record of asynchronous work not yet seen complete (parity or -1)
    int pend_k[2] = {-1, -1}, pend_u[2] = {-1, -1}, pend_s[2] = {-1, -1};
    int ph_k[2] = {0, 0}, ph_u[2] = {0, 0}, ph_s[2] = {0, 0};  // uses of each barrier so far

    auto load_chunk = [&](int e, int cb) {
        const int64_t off = ((int64_t)e * C) % a.src_len;
        const uint32_t bar = smem_u32(&X.bar_k[cb]);
        pend_k[cb] = ph_k[cb] & 1;
        mbar_expect_tx(bar, 2 * T * TILE_BYTES);
        for (int t = 0; t < T; ++t) {
            tma_load_3d(sbase + OFF_K + cb * CHB + t * TILE_BYTES, &tm_k, 0, (int)(off + 128 * t), bh, bar);
            tma_load_3d(sbase + OFF_V + cb * CHB + t * TILE_BYTES, &tm_v, 0, (int)(off + 128 * t), bh, bar);
        }
    };
    auto load_u = [&](int blk, int ub) {
        const uint32_t bar = smem_u32(&X.bar_u[ub]);
        pend_u[ub] = ph_u[ub] & 1;
        mbar_expect_tx(bar, UBUF);
        tma_load_3d(sbase + ub * UBUF, &tm_u, 0, blk * NB, bh, bar);
        tma_load_3d(sbase + ub * UBUF + NB * ROWB, &tm_u, 64, blk * NB, bh, bar);
    };
    // S buffer sb = chunk keys (T tiles) x (u_hi + u_lo) of U buffer ub.  Issuer k takes
    // eight N = 128 MMAs: with one token tile the slot columns [128k, 128k + 128), with two
    // the token tile k; every accumulator element takes the same K-steps in the same order
    auto issue_mma = [&](int cb, int ub, int sb, int k) {
        tc_fence_after();
        const int t = T == 1 ? 0 : k, c0 = T == 1 ? 128 * k : 0;
        for (int ks = 0; ks < 4; ++ks)
            for (int pt = 0; pt < 2; ++pt) {
                const uint64_t ad = sdesc_sw128(sbase + OFF_K + cb * CHB + t * TILE_BYTES + ks * 32, 16, 1024);
                const uint64_t bd =
                    sdesc_sw128(sbase + ub * UBUF + (pt * NB + c0) * ROWB + ks * 32, 16, 1024);
                mma_bf16_ss(tmem + 256 * sb + t * NB + c0, ad, bd, idesc, (ks | pt) ? 1u : 0u);
            }
        mma_commit(smem_u32(&X.bar_s[sb]));
        pend_s[sb] = ph_s[sb] & 1;
    };
    auto wait_bar = [&](unsigned long long* bar, int& ph, int* pend) -> bool {
        const bool ok = mbar_wait(smem_u32(bar), ph & 1, &X.abort_flag, a.status);
        if (ok && pend) *pend = -1;
        ++ph;
        return ok;
    };

    if (tid == 0 && a.e_begin < a.e_end && !a.test_stall) load_chunk(a.e_begin, 0);
    bool fail = false;
    // gates are loaded one event ahead (off the chain): thread 2t holds token t's
    auto gate_of = [&](int e) -> float {
        const int t = tid >> 1;
        return ((tid & 1) == 0 && t < C && e < a.e_end)
                   ? a.g_src[(int64_t)bh * a.src_row + ((int64_t)e * C) % a.src_len + t]
                   : 0.0f;
    };
    float g_nx = gate_of(a.e_begin);
    // snapshot of the read view after event snap_e (n rows); the copy is made before the
    // next event's owners rewrite the view, at the barrier that ends its set-up
    int snap_e = -1, snap_n = 0;
    auto snapshot = [&]() {
        if (a.snap_k && !a.log_k && snap_e >= 0 && snap_e < a.snap_events) {
            // full snapshot rows: the compact key rows behind zeros on the leading pieces
            const int64_t base = ((int64_t)bh * a.snap_events + snap_e) * M * ROWB;
            const int nchunks = snap_n * 8;
            const uint4* sk4 = reinterpret_cast<const uint4*>(g_vk);
            const uint4* sv4 = reinterpret_cast<const uint4*>(g_vv);
            uint4* dk4 = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(a.snap_k) + base);
            uint4* dv4 = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(a.snap_v) + base);
            for (int i = tid; i < nchunks; i += NT) {
                const int row = i >> 3, pc = i & 7;
                const uint4 wk = pc < zc ? make_uint4(0u, 0u, 0u, 0u) : sk4[row * (8 - zc) + pc - zc];
                const uint4 wv = sv4[i];
                dk4[i] = wk;
                dv4[i] = wv;
            }
        }
        snap_e = -1;
    };
    KVM_PROBE_DECL(16)
    KVM_PROBE_START()
    for (int e = a.e_begin, it = 0; e < a.e_end; ++e, ++it) {
        const int cb = it & 1;
        const Sched sc = a.sched ? a.sched[e] : a.sched0;
        const int64_t first_pos = (int64_t)e * C;
        const int n0 = sc.n0, na = sc.a;
        const int nb = n0 > S ? (n0 + NB - 1) / NB : 0;
        const uint8_t* kch = sm + OFF_K + cb * CHB;
        const uint8_t* vch = sm + OFF_V + cb * CHB;
        const float g_here = g_nx;
        if (!wait_bar(&X.bar_k[cb], ph_k[cb], tid == 0 ? &pend_k[cb] : nullptr)) fail = true;
        g_nx = gate_of(e + 1);
        KVM_PROBE_LAP(0)
#ifdef KVM_PROBE
        probe_acc[15] += 1;
#endif
        if (tid == 0) {
            // the next chunk loads into the buffer the previous event finished with
            if (!fail && e + 1 < a.e_end) load_chunk(e + 1, cb ^ 1);
            if (!fail && nb > 0) {
                load_u(0, 0);
                if (nb > 1) load_u(1, 1);
            }
        }
        // per-token set-up: gates, key norms (two threads per token), kinds
        {
            const int t = tid >> 1, h = tid & 1;
            if (tid < 2 * C) {
                float ss = 0.0f;
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    const int row = t & 127;
                    const uint4 w = *reinterpret_cast<const uint4*>(kch + (t >> 7) * TILE_BYTES + swz(row, 4 * h + ch));
                    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float2 f = unpack2(wv[u]);
                        ss = fmaf(f.x, f.x, ss);
                        ss = fmaf(f.y, f.y, ss);
                    }
                }
                ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                if (h == 0) {
                    X.g[t] = g_here;
                    X.kn[t] = sqrtf(ss);
                    const bool sink = first_pos + t < S;
                    X.kind[t] = sink ? 2 : -1;
                    X.slot[t] = sink ? (int)(first_pos + t) : -1;
                }
            }
            for (int i = tid; i < (M + 31) / 32; i += NT) X.slotbits[i] = 0u;
            for (int i = tid; i < MAXC * (MAXC / 32) / 4; i += NT)
                reinterpret_cast<uint4*>(&X.tmask[0][0])[i] = make_uint4(0, 0, 0, 0);
            if (tid < MAXC) X.kfound[tid] = -1;
        }
        snapshot();
        // the first block's directions have been loading during the set-up
        if (issuer && !fail && nb > 0) {
            if (!wait_bar(&X.bar_u[0], ph_u[0], tid == 0 ? &pend_u[0] : nullptr)) fail = true;
            else issue_mma(cb, 0, 0, ik);
        }
        if (__syncthreads_or(fail)) break;
        KVM_PROBE_LAP(1)

        // similarity blocks: MMA of block b + 1 runs while block b is scanned
        float best = -INFINITY, sec = -INFINITY;
        int barg = -1;
        for (int b = 0; b < nb; ++b) {
            const int sb = b & 1;
            if (issuer && b + 1 < nb) {
                if (!wait_bar(&X.bar_u[(b + 1) & 1], ph_u[(b + 1) & 1], tid == 0 ? &pend_u[(b + 1) & 1] : nullptr))
                    fail = true;
                else
                    issue_mma(cb, (b + 1) & 1, (b + 1) & 1, ik);
            }
            const bool ok = wait_bar(&X.bar_s[sb], ph_s[sb], issuer ? &pend_s[sb] : nullptr);
            fail = fail || !ok;
            tc_fence_after();
            // U buffer sb is free once this block's MMA completed
            if (tid == 0 && !fail && b + 2 < nb) load_u(b + 2, sb);
            if (!__any_sync(0xffffffffu, fail)) {
                uint32_t va[32], vb[32];
                const uint32_t ta = tmem + lane_base + 256 * sb + 64 * G;
                tmem_ld32(ta, va);
                tmem_ld32(ta + 32, vb);
                tmem_wait_ld();
                if (tok < C) {
                    const int base = b * NB + colslot;
                    scan32<GAP>(va, base, S, n0, best, sec, barg);
                    scan32<GAP>(vb, base + 32, S, n0, best, sec, barg);
                }
            }
            tc_fence_before();
            if (__syncthreads_or(fail)) {
                fail = true;
                break;
            }
        }
        if (fail) break;
        KVM_PROBE_LAP(2)
        if (tok < C) {
            X.pb[part][tok] = best;
            X.ps[part][tok] = sec;
            X.pa[part][tok] = barg;
        }
        __syncthreads();
        // combine the partials of each token; surprise score m_t
        best = -INFINITY;
        sec = -INFINITY;
        barg = -1;
        const bool cand = tid < C && X.kind[tid] != 2;
        if (cand && nb > 0)
            for (int p = 0; p < nparts; ++p) combine(best, sec, barg, X.pb[p][tid], X.ps[p][tid], X.pa[p][tid]);
        const float kn = tid < C ? X.kn[tid] : 0.0f;
        if (cand) X.m[tid] = barg < 0 ? -INFINITY : (kn > 0.0f ? best / kn : 0.0f);
        else if (tid < C) X.m[tid] = INFINITY;  // sinks are never append candidates
        __syncthreads();
        KVM_PROBE_LAP(3)

        // surprise selection: the a lowest scores (ties to the lower position) are appended
        if (na > 0) {
            // rank = candidates with a smaller score (ties: lower position); only whether
            // it is below a matters, so the count stops there
            int rank = 0;
            if (cand) {
                const float mt = X.m[tid];
                for (int u0 = 0; u0 < C && rank < na; u0 += 8) {  // C is a multiple of 16
                    const float4 m0 = *reinterpret_cast<const float4*>(&X.m[u0]);
                    const float4 m1 = *reinterpret_cast<const float4*>(&X.m[u0 + 4]);
                    const float mu[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
                    for (int i = 0; i < 8; ++i) rank += (mu[i] < mt) || (mu[i] == mt && u0 + i < tid);
                }
            }
            KVM_PROBE_LAP(9)
            const bool app = cand && rank < na;
            // appended slots in position order: warp ballots and their prefix
            unsigned bal = 0;
            if (warp < (C + 31) / 32) {
                bal = __ballot_sync(0xffffffffu, app);
                if (lane == 0) X.wapp[warp] = __popc(bal);
            }
            __syncthreads();
            if (cand) X.kind[tid] = app ? 1 : 0;
            if (app) {
                int before = __popc(bal & ((1u << lane) - 1u));
                for (int w = 0; w < warp; ++w) before += X.wapp[w];
                X.slot[tid] = n0 + before;
            }
            __syncthreads();
            KVM_PROBE_LAP(10)
            // directions of the new slots (one warp each, from g * k of the founding
            // token), staged as fp32 hi + lo in the U area and written to the workspace
            float* ustage = reinterpret_cast<float*>(sm);
            for (int t = warp; t < C; t += NW) {
                if (X.kind[t] != 1) continue;
                const int jn = X.slot[t];
                const float g = X.g[t];
                const float2 kk = row_pair(kch + (t >> 7) * TILE_BYTES, t & 127, lane);
                float2 c;
                uint32_t hw, lw;
                warp_dir(make_float2(g * kk.x, g * kk.y), lane, g_u + (int64_t)jn * 128, c, hw, lw);
                const float2 hf = unpack2(hw), lf = unpack2(lw);
                reinterpret_cast<float2*>(ustage + (jn - n0) * D)[lane] = make_float2(hf.x + lf.x, hf.y + lf.y);
            }
            __syncthreads();
            KVM_PROBE_LAP(11)
            // the remaining tokens also compare against the new slots
            if (tid < C && X.kind[tid] == 0) {
                float kx[64];
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const uint4 w = *reinterpret_cast<const uint4*>(kch + (tid >> 7) * TILE_BYTES + swz(tid & 127, ch));
                    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float2 f = unpack2(wv[u]);
                        kx[ch * 8 + 2 * u] = f.x;
                        kx[ch * 8 + 2 * u + 1] = f.y;
                    }
                }
                for (int jj = 0; jj < na; ++jj) {
                    const float4* ur = reinterpret_cast<const float4*>(ustage + jj * D);
                    float p[8];
#pragma unroll
                    for (int x4 = 0; x4 < 16; ++x4) {
                        const float4 u4 = ur[x4];
                        if (x4 < 2) {
                            p[4 * x4] = kx[4 * x4] * u4.x;
                            p[4 * x4 + 1] = kx[4 * x4 + 1] * u4.y;
                            p[4 * x4 + 2] = kx[4 * x4 + 2] * u4.z;
                            p[4 * x4 + 3] = kx[4 * x4 + 3] * u4.w;
                        } else {
                            const int o = (4 * x4) & 7;
                            p[o] = fmaf(kx[4 * x4], u4.x, p[o]);
                            p[o + 1] = fmaf(kx[4 * x4 + 1], u4.y, p[o + 1]);
                            p[o + 2] = fmaf(kx[4 * x4 + 2], u4.z, p[o + 2]);
                            p[o + 3] = fmaf(kx[4 * x4 + 3], u4.w, p[o + 3]);
                        }
                    }
                    const float s = ((p[0] + p[1]) + (p[2] + p[3])) + ((p[4] + p[5]) + (p[6] + p[7]));
                    const int jn = n0 + jj;
                    if (s > best) {
                        sec = best;
                        best = s;
                        barg = jn;
                    } else if (s > sec) {
                        sec = s;
                    }
                }
            }
        } else if (cand) {
            X.kind[tid] = 0;
        }
        KVM_PROBE_LAP(4)
        if (tid < C && X.kind[tid] == 0) {
            X.slot[tid] = barg;
            if (barg < 0 && a.status) atomicOr(a.status, STATUS_DEVICE);
        }
        if (tid < C && e < a.dbg_events) {
            const int64_t o = ((int64_t)bh * a.dbg_events + e) * C + tid;
            const int kd = X.kind[tid];
            if (a.dbg_assign) a.dbg_assign[o] = X.slot[tid];
            if (a.dbg_kind) a.dbg_kind[o] = kd;
            if (a.dbg_m) a.dbg_m[o] = kd == 2 ? __int_as_float(0x7fc00000) : X.m[tid];
            if (GAP && a.dbg_gap) {
                float gp = __int_as_float(0x7fc00000);
                if (kd == 0) gp = sec == -INFINITY ? INFINITY : (kn > 0.0f ? (best - sec) / kn : 0.0f);
                a.dbg_gap[o] = gp;
            }
        }
        // touched slots: bitmap, then compact indices in slot order
        if (tid < C && X.slot[tid] >= 0 && !kvm_check(X.slot[tid] < sc.n_after, a.status)) X.slot[tid] = -1;
        if (tid < C && X.slot[tid] >= 0) atomicOr(&X.slotbits[X.slot[tid] >> 5], 1u << (X.slot[tid] & 31));
        __syncthreads();
        const int nwords = (sc.n_after + 31) / 32;
        if (warp == 0) {
            int cnts[4], tot = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int w = lane * 4 + i;
                cnts[i] = w < nwords ? __popc(X.slotbits[w]) : 0;
                tot += cnts[i];
            }
            int incl = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            int run = incl - tot;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                X.wbase[lane * 4 + i] = run;
                run += cnts[i];
            }
            if (lane == 31) X.wbase[MAXM / 32] = run;
        }
        __syncthreads();
        if (tid < C && X.slot[tid] >= 0) {
            const int s = X.slot[tid];
            const int k = X.wbase[s >> 5] + __popc(X.slotbits[s >> 5] & ((1u << (s & 31)) - 1u));
            X.tslot[k] = s;
            if (X.kind[tid] == 0) atomicOr(&X.tmask[k][tid >> 5], 1u << (tid & 31));
            else X.kfound[k] = tid;
        }
        __syncthreads();
        const int ntouched = X.wbase[MAXM / 32];
        if (tid == 0 && a.log_k && e < a.snap_events) a.log_cnt[(int64_t)bh * a.snap_events + e] = ntouched;
        KVM_PROBE_LAP(5)

        // owners: eight lanes per touched slot (dims 8 sl .. 8 sl + 7 on sub-lane sl), so
        // a warp works on four slots at a time; reductions over the eight lanes
        {
            const int grp = lane >> 3, sl = lane & 7;
            // the state of a round's slots is loaded one round ahead (global-memory latency)
            float4 nk0 = make_float4(0.f, 0.f, 0.f, 0.f), nk1 = nk0, nv0 = nk0, nv1 = nk0;
            int ncnt = 0;
            float nrho = 0.0f;
            auto load_round = [&](int kk) {
                if (kk < ntouched && X.kfound[kk] < 0) {
                    const int jj = X.tslot[kk];
                    const float4* pk = reinterpret_cast<const float4*>(g_sk + (int64_t)jj * D + 8 * sl);
                    const float4* pv = reinterpret_cast<const float4*>(g_sv + (int64_t)jj * D + 8 * sl);
                    nk0 = pk[0];
                    nk1 = pk[1];
                    nv0 = pv[0];
                    nv1 = pv[1];
                    ncnt = g_cnt[jj];
                    nrho = g_rho[jj];
                }
            };
            load_round(4 * warp + grp);
            for (int k = 4 * warp + grp; k - grp < ntouched; k += 4 * NW) {
                const bool act = k < ntouched;
                const int j = act ? X.tslot[k] : 0;
                const int ft = act ? X.kfound[k] : -1;
                float xk[8] = {nk0.x, nk0.y, nk0.z, nk0.w, nk1.x, nk1.y, nk1.z, nk1.w};
                float xv[8] = {nv0.x, nv0.y, nv0.z, nv0.w, nv1.x, nv1.y, nv1.z, nv1.w};
                int cnt = ncnt;
                float rho = nrho;
                load_round(k + 4 * NW);
                // a token's eight dims of this sub-lane: one 16-byte swizzled chunk
                auto chunk8 = [&](const uint8_t* base, int t, float (&y)[8]) {
                    const uint4 w = *reinterpret_cast<const uint4*>(base + (t >> 7) * TILE_BYTES + swz(t & 127, sl));
                    const float2 a0 = unpack2(w.x), a1 = unpack2(w.y), a2 = unpack2(w.z), a3 = unpack2(w.w);
                    y[0] = a0.x; y[1] = a0.y; y[2] = a1.x; y[3] = a1.y;
                    y[4] = a2.x; y[5] = a2.y; y[6] = a3.x; y[7] = a3.y;
                };
                float vsq = 0.0f;
                if (act && ft >= 0) {
                    const float gf = X.g[ft];
                    float kk[8], vv[8];
                    chunk8(kch, ft, kk);
                    chunk8(vch, ft, vv);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        xk[i] = gf * kk[i];
                        xv[i] = gf * vv[i];
                        vsq = fmaf(vv[i], vv[i], vsq);
                    }
                    cnt = 1;
                }
                // |v| of a founding token (read radius), over the group's eight lanes
                vsq += __shfl_xor_sync(0xffffffffu, vsq, 1);
                vsq += __shfl_xor_sync(0xffffffffu, vsq, 2);
                vsq += __shfl_xor_sync(0xffffffffu, vsq, 4);
                if (act && ft >= 0) rho = sqrtf(vsq);
                // merged tokens in position order
                if (act) {
                    // one loop over the set bits of all mask words (a warp runs as many
                    // rounds as its busiest slot has tokens)
                    const int nw = (C + 31) / 32;
                    int w8 = 0;
                    uint32_t m = X.tmask[k][0];
                    while (true) {
                        while (m == 0u && ++w8 < nw) m = X.tmask[k][w8];
                        if (w8 >= nw) break;
                        {
                            const int t = (w8 << 5) + __ffs(m) - 1;
                            m &= m - 1;
                            const float gt = X.g[t];
                            float kk[8], vv[8];
                            chunk8(kch, t, kk);
                            chunk8(vch, t, vv);
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                xk[i] = fmaf(gt, kk[i], xk[i]);
                                xv[i] = fmaf(gt, vv[i], xv[i]);
                            }
                            ++cnt;
                        }
                    }
                }
                __syncwarp();
                // centred key, its norm, and the value norm: sums over the group's lanes
                float s1 = 0.0f, sv = 0.0f;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    s1 += xk[i];
                    sv = fmaf(xv[i], xv[i], sv);
                }
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) {
                    s1 += __shfl_xor_sync(0xffffffffu, s1, o);
                    sv += __shfl_xor_sync(0xffffffffu, sv, o);
                }
                const float mean = s1 * (1.0f / 64.0f);
                float c[8], ss = 0.0f;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    c[i] = xk[i] - mean;
                    ss = fmaf(c[i], c[i], ss);
                }
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                if (act) {
                    float4* qk = reinterpret_cast<float4*>(g_sk + (int64_t)j * D + 8 * sl);
                    float4* qv = reinterpret_cast<float4*>(g_sv + (int64_t)j * D + 8 * sl);
                    qk[0] = make_float4(xk[0], xk[1], xk[2], xk[3]);
                    qk[1] = make_float4(xk[4], xk[5], xk[6], xk[7]);
                    qv[0] = make_float4(xv[0], xv[1], xv[2], xv[3]);
                    qv[1] = make_float4(xv[4], xv[5], xv[6], xv[7]);
                    if (sl == 0) {
                        g_cnt[j] = cnt;
                        g_rho[j] = rho;
                    }
                    // direction u = c / |c| as bf16 hi + lo; read key LayerNorm(sum / count) =
                    // c / sqrt(|c|^2 / 64 + eps count^2) with the rotary dims zeroed; read value
                    // rho * unit(sum_v) (or sum_v / count)
                    const float inv = ss > 0.0f ? 1.0f / sqrtf(ss) : 0.0f;
                    const float fc = (float)cnt;
                    const float rs = 1.0f / sqrtf(ss * (1.0f / 64.0f) + a.ln_eps * fc * fc);
                    const float nv = sqrtf(sv);
                    const float f = a.no_vnorm ? 1.0f / fc : (nv > 0.0f ? rho / nv : 0.0f);
                    uint32_t hi[4], lo[4], wk[4], wv[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float u0 = c[2 * i] * inv, u1 = c[2 * i + 1] * inv;
                        hi[i] = pack2(u0, u1);
                        const float2 hf = unpack2(hi[i]);
                        lo[i] = pack2(u0 - hf.x, u1 - hf.y);
                        const int d0 = 8 * sl + 2 * i;
                        wk[i] = pack2(d0 < a.r ? 0.0f : c[2 * i] * rs, d0 + 1 < a.r ? 0.0f : c[2 * i + 1] * rs);
                        wv[i] = pack2(xv[2 * i] * f, xv[2 * i + 1] * f);
                    }
                    uint4* urow = reinterpret_cast<uint4*>(g_u + (int64_t)j * 128);
                    urow[sl] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    urow[8 + sl] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    if (sl >= zc)
                        reinterpret_cast<uint4*>(g_vk + (int64_t)j * DK)[sl - zc] = make_uint4(wk[0], wk[1], wk[2], wk[3]);
                    reinterpret_cast<uint4*>(g_vv + (int64_t)j * D)[sl] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                    if (a.log_k && e < a.snap_events) {
                        // the touched row, full width (zeros on the rotary dims), into the event's log
                        const int64_t lrow = ((int64_t)bh * a.snap_events + e) * C + k;
                        reinterpret_cast<uint4*>(a.log_k)[lrow * 8 + sl] = make_uint4(wk[0], wk[1], wk[2], wk[3]);
                        reinterpret_cast<uint4*>(a.log_v)[lrow * 8 + sl] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                        if (sl == 0) a.log_idx[lrow] = j;
                    }
                }
            }
        }
        KVM_PROBE_LAP(6)
        // the next event's TMA reads the directions written above
        fence_proxy_async_all();
        __syncthreads();
        KVM_PROBE_LAP(7)
        n = sc.n_after;
        // this event's snapshot is copied while the next event sets up
        snap_e = e;
        snap_n = n;
        KVM_PROBE_LAP(8)
    }
    if (!fail) snapshot();

    if (tid == 0) KVM_PROBE_FLUSH(g_probe_big, 0, 16)
    // after an abort: let the copies and MMAs this CTA issued land before its shared
    // and tensor memory are released (each wait bounded; they depend on nothing else)
    if (issuer && X.abort_flag) {
        auto drain = [&](unsigned long long* bar, int parity) {
            if (parity < 0) return;
            const long long t0 = clock64();
            while (!mbar_try(smem_u32(bar), (uint32_t)parity) && clock64() - t0 < (1ll << 28)) {
            }
        };
        for (int i = 0; i < 2; ++i) {
            if (tid == 0) {
                drain(&X.bar_k[i], pend_k[i]);
                drain(&X.bar_u[i], pend_u[i]);
            }
            drain(&X.bar_s[i], pend_s[i]);  // each issuer: the MMAs it issued
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace foldbig

KVM_PROBE_READOUT(kvm_probe_read_big, foldbig::g_probe_big)

bool fold_big_supported(const FoldArgs& a, bool bf16) {
    return bf16 && a.C >= 16 && a.C <= foldbig::MAXC && a.M <= foldbig::MAXM;
}

namespace foldbig {
// One CTA per (row, slot range) walks the events in order: snapshot e takes, for each
// slot of its range below n_after(e), the row event e logged for it, else the row of
// snapshot e - 1 (a slot new at e is always logged: founding touches it).
constexpr int RB_T = 256;        // threads
constexpr int RB_SLOTS = 256;    // slots per CTA
__global__ void __launch_bounds__(RB_T) snap_rebuild_kernel(const SnapRebuildArgs a) {
    __shared__ int inv[RB_SLOTS];
    const int tid = threadIdx.x;
    const int splits = (a.M + RB_SLOTS - 1) / RB_SLOTS;
    const int bh = blockIdx.x / splits;
    const int j0 = (blockIdx.x % splits) * RB_SLOTS;
    if (bh >= a.BH) return;
    for (int i = tid; i < RB_SLOTS; i += RB_T) inv[i] = -1;
    const uint4* lk = reinterpret_cast<const uint4*>(a.log_k);
    const uint4* lv = reinterpret_cast<const uint4*>(a.log_v);
    uint4* sk = reinterpret_cast<uint4*>(a.snap_k);
    uint4* sv = reinterpret_cast<uint4*>(a.snap_v);
    __syncthreads();
    for (int e = a.e_begin; e < a.e_end; ++e) {
        const int64_t ev = (int64_t)bh * a.snap_events + e;
        int cnt = a.log_cnt[ev];
        cnt = cnt < 0 ? 0 : (cnt > a.C ? a.C : cnt);
        const int* idx = a.log_idx + ev * a.C;
        for (int i = tid; i < cnt; i += RB_T) {
            const int j = idx[i];
            if (j >= j0 && j < j0 + RB_SLOTS) inv[j - j0] = i;
        }
        __syncthreads();
        const int n = a.sched[e].n_after;
        const int j1 = n < j0 + RB_SLOTS ? n : j0 + RB_SLOTS;
        const int64_t dst = ev * a.M * 8, prev = (ev - 1) * a.M * 8, lrow = ev * a.C * 8;
        for (int q = tid; q < (j1 - j0) * 8; q += RB_T) {
            const int j = j0 + (q >> 3), pc = q & 7;
            const int i = inv[j - j0];
            uint4 wk = make_uint4(0u, 0u, 0u, 0u), wv = wk;
            if (i >= 0) {
                wk = lk[lrow + (int64_t)i * 8 + pc];
                wv = lv[lrow + (int64_t)i * 8 + pc];
            } else if (e > 0) {
                wk = sk[prev + (int64_t)j * 8 + pc];
                wv = sv[prev + (int64_t)j * 8 + pc];
            }
            sk[dst + (int64_t)j * 8 + pc] = wk;
            sv[dst + (int64_t)j * 8 + pc] = wv;
        }
        __syncthreads();
        for (int i = tid; i < cnt; i += RB_T) {
            const int j = idx[i];
            if (j >= j0 && j < j0 + RB_SLOTS) inv[j - j0] = -1;
        }
        __syncthreads();
    }
}
}  // namespace foldbig

cudaError_t launch_snap_rebuild(const SnapRebuildArgs& a, cudaStream_t s) {
    using namespace foldbig;
    if (a.e_begin >= a.e_end || a.BH == 0) return cudaSuccess;
    const int splits = (a.M + RB_SLOTS - 1) / RB_SLOTS;
    snap_rebuild_kernel<<<a.BH * splits, RB_T, 0, s>>>(a);
    return cudaGetLastError();
}

bool fold_logs_rows(const FoldArgs& a, bool bf16) {
    return !fold_tc_supported(a, bf16) && fold_big_supported(a, bf16);
}

cudaError_t launch_fold_big(const FoldArgs& a, cudaStream_t s) {
    using namespace foldbig;
    const int T = a.C > 128 ? 2 : 1;
    const int NB = 256 / T;
    CUtensorMap mk, mv, mu;
    if (!make_tmap_bf16_3d(&mk, a.k_src, (uint64_t)a.src_row, (uint64_t)a.BH, 128) ||
        !make_tmap_bf16_3d(&mv, a.v_src, (uint64_t)a.src_row, (uint64_t)a.BH, 128) ||
        !make_tmap_bf16_rows(&mu, a.simdir, 128, (uint64_t)a.M, (uint64_t)a.BH, (uint32_t)NB))
        return cudaErrorInvalidValue;
    auto kern = a.dbg_gap ? fold_big_kernel<true> : fold_big_kernel<false>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    kern<<<a.BH, NT, SMEM_BYTES, s>>>(mk, mv, mu, a);
    return cudaGetLastError();
}

}  // namespace kvm
