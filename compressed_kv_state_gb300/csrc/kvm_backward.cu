// Backward of the KVM prefill for chunk-parallel training.
//
// "Key-Value Means" (gist.science technical summary), Contributions and
// Significance: the layer trains chunk-parallel; the pages do not say how the
// gradient passes the winner-take-all assignment.  Reading taken here: the
// fold's discrete decisions (each merged token's slot, the surprise-selected
// appends, the sinks) are constants from the forward pass, read from its
// debug record; the gradient flows through the attention (Core mechanism 4),
// the just-in-time read of the state (Core mechanisms 2 and 4: LayerNorm of
// sum_k / count with the rotary dims zeroed, rho * unit(sum_v)), the
// gate-weighted member sums (Core mechanism 2) and the founders' read radius
// rho = |v| (Core mechanism 3).
//
// Chunks a multiple of 64 take a tiled path for the five attention products: on tcgen05
// (kvm_backward_tc.cu) for bf16 layers with chunks a multiple of 128 whose forward kept
// its log2-sum-exp; otherwise bwd_tile_tc (mma.sync, bf16) or bwd_tile (fp32 FMA), with
// 64-query tiles and 64-key blocks in shared memory.  The row kernels below serve the
// other chunk sizes (one warp per query, key or state row, lanes over the 64 dims, two
// each).  bwd_rotate, bwd_members and bwd_sweep16 serve every path:
//   bwd_rotate   q and k rotated at their own positions (scratch)
//   bwd_stats    per query: log2-sum-exp of its scores and D = dout . out
//   bwd_dq       per query: dq (state part in plain coordinates, window part
//                rotated back)
//   bwd_dkv_win  per key: dk (rotated back) and dv from the queries whose
//                window holds it; dgate = 0
//   bwd_dstate   per fold event and slot: the gradient of the event's read
//                rows (key and value) from the chunk that reads them
//   bwd_members  per (batch, head) row: every slot's member tokens in replay order
//   bwd_sweep16  per slot, half a warp: replays the slot with the recorded decisions
//                (the forward's fp32 sums, in its order), turns each event's read-row
//                gradients into sum and radius gradients (LayerNorm and normalisation
//                backward), and gives each member their sum from its own event to the
//                last (total minus running sum), adding the tokens' k, v and gate
//                gradients.
#include "kvm_internal.cuh"

namespace kvm {
namespace {

constexpr int BW_WARPS = 8;  // warps per CTA of the per-row kernels
constexpr int BW_THREADS = BW_WARPS * 32;

template <typename T> __device__ __forceinline__ float2 ld2(const T* p);
template <> __device__ __forceinline__ float2 ld2<float>(const float* p) {
    return *reinterpret_cast<const float2*>(p);
}
template <> __device__ __forceinline__ float2 ld2<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
__device__ __forceinline__ float dot2(float2 a, float2 b) { return a.x * b.x + a.y * b.y; }

// Lane l holds dims 2l, 2l + 1 of a rotated row y at position p; returns the same
// dims of R_p^T y (rotate-half pairs (i, i + r/2) on dims [0, r)).  Every lane
// takes part in the shuffles.
__device__ __forceinline__ float2 unrotate2(float2 y, int lane, int64_t p, int r, const float2* rope) {
    const int half = r / 2;
    const int x = 2 * lane;
    const int off = half / 2;  // lanes between a dim and its partner (half is even)
    const bool rot = x < r, low = x < half;
    const int partner = !rot ? lane : (low ? lane + off : lane - off);
    const float ox = __shfl_sync(0xffffffffu, y.x, partner);
    const float oy = __shfl_sync(0xffffffffu, y.y, partner);
    if (!rot) return y;
    const int i0 = low ? x : x - half;
    const float2 c0 = rope[p * half + i0], c1 = rope[p * half + i0 + 1];
    // forward: y_i = x_i c - x_{i+h} s, y_{i+h} = x_{i+h} c + x_i s
    if (low) return make_float2(y.x * c0.x + ox * c0.y, y.y * c1.x + oy * c1.y);
    return make_float2(y.x * c0.x - ox * c0.y, y.y * c1.x - oy * c1.y);
}

// rotated rows of q and k, rounded to the layer's dtype like the forward's rotation
template <typename T>
__global__ void bwd_rotate(BackwardArgs a) {
    const int64_t rows = (int64_t)a.BH * a.N;
    const int half = a.r / 2;
    if constexpr (sizeof(T) == 2) {
        if ((half & 7) == 0) {
            // one thread per 16-byte piece (8 dims) of a row, with its rotate-half partner
            const int hc = half >> 3;
            const uint4* qs = reinterpret_cast<const uint4*>(a.q);
            const uint4* ks = reinterpret_cast<const uint4*>(a.k);
            uint4* qd = reinterpret_cast<uint4*>(a.qr);
            uint4* kd = reinterpret_cast<uint4*>(a.kr);
            for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < rows * 8;
                 i += (int64_t)gridDim.x * blockDim.x) {
                const int64_t rw = i >> 3;
                const int c = (int)(i & 7);
                uint4 wq = qs[i], wk = ks[i];
                if (8 * c < a.r) {
                    const bool low = c < hc;
                    const int64_t pi = rw * 8 + (low ? c + hc : c - hc);
                    const uint4 oq = qs[pi], ok = ks[pi];
                    const float2* tab = a.rope + (rw % a.N) * half + (low ? c : c - hc) * 8;
                    __nv_bfloat162* mq = reinterpret_cast<__nv_bfloat162*>(&wq);
                    __nv_bfloat162* mk = reinterpret_cast<__nv_bfloat162*>(&wk);
                    const __nv_bfloat162* pq = reinterpret_cast<const __nv_bfloat162*>(&oq);
                    const __nv_bfloat162* pk = reinterpret_cast<const __nv_bfloat162*>(&ok);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float2 c0 = tab[2 * u], c1 = tab[2 * u + 1];
                        const float2 a2 = __bfloat1622float2(mq[u]), b2 = __bfloat1622float2(pq[u]);
                        const float2 e2 = __bfloat1622float2(mk[u]), f2 = __bfloat1622float2(pk[u]);
                        mq[u] = low ? __floats2bfloat162_rn(a2.x * c0.x - b2.x * c0.y, a2.y * c1.x - b2.y * c1.y)
                                    : __floats2bfloat162_rn(a2.x * c0.x + b2.x * c0.y, a2.y * c1.x + b2.y * c1.y);
                        mk[u] = low ? __floats2bfloat162_rn(e2.x * c0.x - f2.x * c0.y, e2.y * c1.x - f2.y * c1.y)
                                    : __floats2bfloat162_rn(e2.x * c0.x + f2.x * c0.y, e2.y * c1.x + f2.y * c1.y);
                    }
                }
                qd[i] = wq;
                kd[i] = wk;
            }
            return;
        }
    }
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < rows * D;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = i / D;
        const int x = (int)(i - row * D);
        const int64_t p = row % a.N;
        const T* qs = reinterpret_cast<const T*>(a.q) + row * D;
        const T* ks = reinterpret_cast<const T*>(a.k) + row * D;
        float yq = to_f<T>(qs[x]), yk = to_f<T>(ks[x]);
        if (x < 2 * half) {
            const int i2 = x < half ? x : x - half;
            const float2 cs = a.rope[p * half + i2];
            if (x < half) {
                yq = yq * cs.x - to_f<T>(qs[x + half]) * cs.y;
                yk = yk * cs.x - to_f<T>(ks[x + half]) * cs.y;
            } else {
                yq = yq * cs.x + to_f<T>(qs[x - half]) * cs.y;
                yk = yk * cs.x + to_f<T>(ks[x - half]) * cs.y;
            }
        }
        reinterpret_cast<T*>(a.qr)[i] = from_f<T>(yq);
        reinterpret_cast<T*>(a.kr)[i] = from_f<T>(yk);
    }
}

template <typename T>
__global__ void bwd_stats(BackwardArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (w >= (int64_t)a.BH * a.N) return;
    const int bh = (int)(w / a.N);
    const int64_t p = w % a.N;
    const int Wc = a.W / a.C;
    const int64_t c = p / a.C, e = c - Wc - 1, ws = c - Wc > 0 ? (c - Wc) * a.C : 0;
    const int64_t row = (int64_t)bh * a.N;
    const float2 qv = ld2<T>(reinterpret_cast<const T*>(a.q) + (row + p) * D + 2 * lane);
    const float2 qrv = ld2<T>(reinterpret_cast<const T*>(a.qr) + (row + p) * D + 2 * lane);
    float m = -INFINITY, l = 0.0f;
    auto add = [&](float s) {
        const float mn = fmaxf(m, s);
        l = l * exp2f(m - mn) + exp2f(s - mn);
        m = mn;
    };
    if (e >= 0) {
        const int n = a.sched[e].n_after;
        const T* kh = reinterpret_cast<const T*>(a.snap_k) + ((int64_t)bh * a.snap_events + e) * a.M * D;
        for (int j = 0; j < n; ++j) add(warp_sum(dot2(qv, ld2<T>(kh + (int64_t)j * D + 2 * lane))) * a.scale_log2);
    }
    const T* kr = reinterpret_cast<const T*>(a.kr) + row * D;
    for (int64_t t = ws; t <= p; ++t) add(warp_sum(dot2(qrv, ld2<T>(kr + t * D + 2 * lane))) * a.scale_log2);
    const float2 o = ld2<T>(reinterpret_cast<const T*>(a.out) + (row + p) * D + 2 * lane);
    const float2 go = ld2<T>(reinterpret_cast<const T*>(a.dout) + (row + p) * D + 2 * lane);
    const float dd = warp_sum(dot2(o, go));
    if (lane == 0) {
        a.lse[row + p] = m + log2f(l);
        a.dd[row + p] = dd;
    }
}

template <typename T>
__global__ void bwd_dq(BackwardArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (w >= (int64_t)a.BH * a.N) return;
    const int bh = (int)(w / a.N);
    const int64_t p = w % a.N;
    const int Wc = a.W / a.C;
    const int64_t c = p / a.C, e = c - Wc - 1, ws = c - Wc > 0 ? (c - Wc) * a.C : 0;
    const int64_t row = (int64_t)bh * a.N;
    const float2 qv = ld2<T>(reinterpret_cast<const T*>(a.q) + (row + p) * D + 2 * lane);
    const float2 qrv = ld2<T>(reinterpret_cast<const T*>(a.qr) + (row + p) * D + 2 * lane);
    const float2 go = ld2<T>(reinterpret_cast<const T*>(a.dout) + (row + p) * D + 2 * lane);
    const float L = a.lse[row + p], Dp = a.dd[row + p];
    float2 acc_s = make_float2(0.f, 0.f), acc_w = make_float2(0.f, 0.f);
    if (e >= 0) {
        const int n = a.sched[e].n_after;
        const int64_t plane = ((int64_t)bh * a.snap_events + e) * a.M * D;
        const T* kh = reinterpret_cast<const T*>(a.snap_k) + plane;
        const T* vh = reinterpret_cast<const T*>(a.snap_v) + plane;
        for (int j = 0; j < n; ++j) {
            const float2 kx = ld2<T>(kh + (int64_t)j * D + 2 * lane);
            const float P = exp2f(warp_sum(dot2(qv, kx)) * a.scale_log2 - L);
            const float dS = P * (warp_sum(dot2(go, ld2<T>(vh + (int64_t)j * D + 2 * lane))) - Dp);
            acc_s.x = fmaf(dS, kx.x, acc_s.x);
            acc_s.y = fmaf(dS, kx.y, acc_s.y);
        }
    }
    const T* kr = reinterpret_cast<const T*>(a.kr) + row * D;
    const T* vv = reinterpret_cast<const T*>(a.v) + row * D;
    for (int64_t t = ws; t <= p; ++t) {
        const float2 kx = ld2<T>(kr + t * D + 2 * lane);
        const float P = exp2f(warp_sum(dot2(qrv, kx)) * a.scale_log2 - L);
        const float dS = P * (warp_sum(dot2(go, ld2<T>(vv + t * D + 2 * lane))) - Dp);
        acc_w.x = fmaf(dS, kx.x, acc_w.x);
        acc_w.y = fmaf(dS, kx.y, acc_w.y);
    }
    const float2 uw = unrotate2(acc_w, lane, p, a.r, a.rope);
    const float is = a.inv_sqrt_d;
    reinterpret_cast<float2*>(a.dq + (row + p) * D)[lane] = make_float2((uw.x + acc_s.x) * is, (uw.y + acc_s.y) * is);
}

template <typename T>
__global__ void bwd_dkv_win(BackwardArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (w >= (int64_t)a.BH * a.N) return;
    const int bh = (int)(w / a.N);
    const int64_t t = w % a.N;
    const int Wc = a.W / a.C;
    const int64_t ct = t / a.C;
    const int64_t pend = (ct + Wc + 1) * a.C < a.N ? (ct + Wc + 1) * a.C : a.N;  // queries t .. pend-1
    const int64_t row = (int64_t)bh * a.N;
    const float2 kx = ld2<T>(reinterpret_cast<const T*>(a.kr) + (row + t) * D + 2 * lane);
    const float2 vx = ld2<T>(reinterpret_cast<const T*>(a.v) + (row + t) * D + 2 * lane);
    const T* qr = reinterpret_cast<const T*>(a.qr) + row * D;
    const T* go = reinterpret_cast<const T*>(a.dout) + row * D;
    float2 ak = make_float2(0.f, 0.f), av = make_float2(0.f, 0.f);
    for (int64_t p = t; p < pend; ++p) {
        const float2 qx = ld2<T>(qr + p * D + 2 * lane);
        const float2 gx = ld2<T>(go + p * D + 2 * lane);
        const float P = exp2f(warp_sum(dot2(qx, kx)) * a.scale_log2 - a.lse[row + p]);
        const float dS = P * (warp_sum(dot2(gx, vx)) - a.dd[row + p]);
        ak.x = fmaf(dS, qx.x, ak.x);
        ak.y = fmaf(dS, qx.y, ak.y);
        av.x = fmaf(P, gx.x, av.x);
        av.y = fmaf(P, gx.y, av.y);
    }
    const float2 uk = unrotate2(ak, lane, t, a.r, a.rope);
    reinterpret_cast<float2*>(a.dk + (row + t) * D)[lane] = make_float2(uk.x * a.inv_sqrt_d, uk.y * a.inv_sqrt_d);
    reinterpret_cast<float2*>(a.dv + (row + t) * D)[lane] = av;
    if (lane == 0) a.dg[row + t] = 0.0f;
}

template <typename T>
__global__ void bwd_dstate(BackwardArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (w >= (int64_t)a.BH * a.E * a.M) return;
    const int j = (int)(w % a.M);
    const int e = (int)((w / a.M) % a.E);
    const int bh = (int)(w / ((int64_t)a.M * a.E));
    if (j >= a.sched[e].n_after) return;
    const int Wc = a.W / a.C;
    const int64_t c = (int64_t)e + Wc + 1;  // the chunk that reads the state after event e
    const int64_t p0 = c * a.C, p1 = (c + 1) * a.C < a.N ? (c + 1) * a.C : a.N;
    const int64_t row = (int64_t)bh * a.N;
    const int64_t vrow = (((int64_t)bh * a.snap_events + e) * a.M + j) * D;
    const float2 kx = ld2<T>(reinterpret_cast<const T*>(a.snap_k) + vrow + 2 * lane);
    const float2 vx = ld2<T>(reinterpret_cast<const T*>(a.snap_v) + vrow + 2 * lane);
    const T* qq = reinterpret_cast<const T*>(a.q) + row * D;
    const T* go = reinterpret_cast<const T*>(a.dout) + row * D;
    float2 ak = make_float2(0.f, 0.f), av = make_float2(0.f, 0.f);
    for (int64_t p = p0; p < p1; ++p) {
        const float2 qx = ld2<T>(qq + p * D + 2 * lane);
        const float2 gx = ld2<T>(go + p * D + 2 * lane);
        const float P = exp2f(warp_sum(dot2(qx, kx)) * a.scale_log2 - a.lse[row + p]);
        const float dS = P * (warp_sum(dot2(gx, vx)) - a.dd[row + p]);
        ak.x = fmaf(dS, qx.x, ak.x);
        ak.y = fmaf(dS, qx.y, ak.y);
        av.x = fmaf(P, gx.x, av.x);
        av.y = fmaf(P, gx.y, av.y);
    }
    const int64_t o = (((int64_t)bh * a.E + e) * a.M + j) * D;
    reinterpret_cast<float2*>(a.dks + o)[lane] = make_float2(ak.x * a.inv_sqrt_d, ak.y * a.inv_sqrt_d);
    reinterpret_cast<float2*>(a.dvs + o)[lane] = av;
}

// Per row, one CTA: every slot's members (the tokens the recorded decisions sent to it)
// as one list in the replay's order: by event, the founder first, then the merged tokens
// in position order.  Entry (t << 2) | kind; slot j's part is mem[moff[j] .. moff[j + 1]).
// A record entry that names no slot of its event or no known kind latches the status
// word and is left out.  The ordered append is serial (one warp), so the whole CTA first
// stages a run of events' entries in shared memory, packed (slot << 2) | kind or -1, and
// the warp reads them there instead of waiting on global loads at every step.
constexpr int MB_THREADS = 256;
constexpr int MB_STAGE = 4096;  // entries staged at a time (>= 16 events of the largest chunk)
__global__ void __launch_bounds__(MB_THREADS) bwd_members(BackwardArgs a) {
    extern __shared__ int cur[];  // [M + 1]: counts, then list cursors; then stage[MB_STAGE]
    int* stage = cur + a.M + 1;
    __shared__ int part[MB_THREADS / 32];
    const int bh = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int C = a.C, M = a.M, E = a.E;
    const int64_t rec0 = (int64_t)bh * a.rec_events * C;
    int* moff = a.moff + (int64_t)bh * (M + 1);
    int* list = a.mem + (int64_t)bh * E * C;
    // kind of entry (e, i) and its slot, or -1 for an invalid entry
    auto entry = [&](int e, int i, int& sj) -> int {
        const int64_t o = rec0 + (int64_t)e * C + i;
        sj = a.assign[o];
        const int kn = a.kind[o];
        return sj >= 0 && sj < a.sched[e].n_after && kn >= 0 && kn <= 2 ? kn : -1;
    };
    for (int j = tid; j <= M; j += MB_THREADS) cur[j] = 0;
    __syncthreads();
    for (int q = tid; q < E * C; q += MB_THREADS) {
        int sj;
        if (entry(q / C, q % C, sj) >= 0)
            atomicAdd(&cur[sj], 1);
        else if (a.status)
            atomicOr(a.status, STATUS_DEVICE);
    }
    __syncthreads();
    // exclusive prefix sum of the counts: each thread a contiguous range of slots
    const int per = (M + MB_THREADS - 1) / MB_THREADS;
    const int j0 = min(M, tid * per), j1 = min(M, j0 + per);
    int own = 0;
    for (int j = j0; j < j1; ++j) own += cur[j];
    int x = own;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) part[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int p = lane < MB_THREADS / 32 ? part[lane] : 0;
#pragma unroll
        for (int d = 1; d < MB_THREADS / 32; d <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, p, d);
            if (lane >= d) p += y;
        }
        if (lane < MB_THREADS / 32) part[lane] = p;
    }
    __syncthreads();
    int run = x - own + (warp > 0 ? part[warp - 1] : 0);
    for (int j = j0; j < j1; ++j) {
        const int c = cur[j];
        cur[j] = run;
        moff[j] = run;
        run += c;
    }
    if (j0 < j1 && j1 == M) moff[M] = run;
    __syncthreads();
    // one warp appends in order: per event the founders, then the merged tokens; lanes of a
    // batch that go to the same slot take consecutive places in lane (= position) order
    const unsigned below = (1u << lane) - 1u;
    const int per_stage = MB_STAGE / C;
    for (int e0 = 0; e0 < E; e0 += per_stage) {
        const int ne = min(per_stage, E - e0);
        for (int q = tid; q < ne * C; q += MB_THREADS) {
            int sj;
            const int kn = entry(e0 + q / C, q % C, sj);
            stage[q] = kn >= 0 ? (sj << 2) | kn : -1;
        }
        __syncthreads();
        if (warp == 0) {
            for (int el = 0; el < ne; ++el)
                for (int pass = 0; pass < 2; ++pass)
                    for (int base = 0; base < C; base += 32) {
                        const int i = base + lane;
                        const int x = i < C ? stage[el * C + i] : -1;
                        const int kn = x >= 0 ? (x & 3) : -1, sj = x >> 2;
                        const bool in = kn >= 0 && (pass == 0 ? kn >= 1 : kn == 0);
                        if (__ballot_sync(0xffffffffu, in) == 0u) continue;  // nothing to place (no founder, say)
                        const unsigned peers = __match_any_sync(0xffffffffu, in ? sj : -1 - lane);
                        int at = 0;
                        if (in) at = cur[sj] + __popc(peers & below);
                        __syncwarp();
                        if (in) {
                            list[at] = (int)((((int64_t)(e0 + el) * C + i) << 2) | kn);
                            if ((peers & below) == 0u) cur[sj] += __popc(peers);
                        }
                        __syncwarp();
                    }
        }
        __syncthreads();
    }
}

// Per slot (every slot's history is its own, so the rows' slots run in parallel): pass 1
// replays the slot through the events with the recorded decisions (its member list: the
// founder first, then its merged tokens in position order: the forward's fp32 sums) and
// turns each event's read-row gradients of the slot into sum and radius gradients
// (LayerNorm and normalisation backward), keeping their running sum over the events.  A
// token that joined at event e is in every state from e on, so its gradient is the sum
// over events >= e: the total at the end of pass 1 minus the running sum before e, which
// pass 1 stores (in the read-row gradient buffers, already consumed there) only at the
// events where some member joined.  Pass 2 then visits each member once.
// Half a warp per slot (two slots a warp; lanes over the dims, four each): the reductions
// take four shuffle levels and each instruction serves two slots.  Every shuffle names only its own half's lanes, which follow their
// slot's control flow together.
template <typename T> __device__ __forceinline__ float4 ld4(const T* p);
template <> __device__ __forceinline__ float4 ld4<float>(const float* p) {
    return *reinterpret_cast<const float4*>(p);
}
template <> __device__ __forceinline__ float4 ld4<__nv_bfloat16>(const __nv_bfloat16* p) {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
    const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}
__device__ __forceinline__ float dot4(float4 a, float4 b) { return (a.x * b.x + a.y * b.y) + (a.z * b.z + a.w * b.w); }
__device__ __forceinline__ float sum4(float4 a) { return (a.x + a.y) + (a.z + a.w); }
__device__ __forceinline__ float half_sum(float v, unsigned hm) {
#pragma unroll
    for (int k = 8; k >= 1; k >>= 1) v += __shfl_xor_sync(hm, v, k);
    return v;
}

// CTAs of two warps: at its 88 registers a thread the sweep fits 23 warps an SM, which
// 256-thread CTAs round down to 16 and 64-thread CTAs to 22
constexpr int SW_WARPS = 2;
template <typename T>
__global__ void __launch_bounds__(SW_WARPS * 32) bwd_sweep16(BackwardArgs a) {
    const int lane = threadIdx.x & 31, hl = lane & 15, hf = lane >> 4;
    const unsigned hm = 0xFFFFu << (16 * hf);
    const int64_t sid = 2 * (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) + hf;
    if (sid >= (int64_t)a.BH * a.M) return;
    const int bh = (int)(sid / a.M);
    const int j = (int)(sid % a.M);
    const int C = a.C, M = a.M, r = a.r;
    const int64_t row = (int64_t)bh * a.N;
    const T* kk = reinterpret_cast<const T*>(a.k) + row * D;
    const T* vv = reinterpret_cast<const T*>(a.v) + row * D;
    const float* gg = a.g + row;
    if (a.E == 0 || j >= a.sched[a.E - 1].n_after) return;  // slot never founded
    const int* lst = a.mem + (int64_t)bh * a.E * C;
    const int m0 = a.moff[(int64_t)bh * (M + 1) + j], m1 = a.moff[(int64_t)bh * (M + 1) + j + 1];
    const int d0 = 4 * hl;  // this lane's dims d0 .. d0 + 3
    // the member list through a window of 16 entries in the half's registers
    int wbase = -64, wbuf = 0;
    auto member = [&](int p, bool fwd) -> int {
        if (p < wbase || p >= wbase + 16) {
            wbase = fwd ? p : max(m0, p - 15);
            wbuf = wbase + hl < m1 ? lst[wbase + hl] : 0;
        }
        return __shfl_sync(hm, wbuf, p - wbase, 16);
    };
    float4 sk = make_float4(0.f, 0.f, 0.f, 0.f), sv = sk;
    int cnt = 0;
    float rho = 0.0f;
    // running sums over the events so far of the slot's sum and radius gradients
    float4 Pk = make_float4(0.f, 0.f, 0.f, 0.f), Pv = Pk;
    float Pr = 0.0f;
    // pass 1
    int ptr = m0;
    for (int e = 0; e < a.E; ++e) {
        const int n = a.sched[e].n_after;
        if (j >= n) continue;  // not founded yet (founding appends at the end)
        const int64_t o = (((int64_t)bh * a.E + e) * M + j) * D + d0;
        // the event's read-row gradients, loaded while the members are replayed
        float4 gkh = *reinterpret_cast<const float4*>(a.dks + o);
        const float4 gvh = *reinterpret_cast<const float4*>(a.dvs + o);
        const int64_t tend = (int64_t)(e + 1) * C;
        bool joined = false;
        while (ptr < m1) {
            const int ent = member(ptr, true);
            const int64_t t = ent >> 2;
            if (t >= tend) break;  // a member of a later event
            ++ptr;
            joined = true;
            const float gt = gg[t];
            const float4 kx = ld4<T>(kk + t * D + d0), vx = ld4<T>(vv + t * D + d0);
            if ((ent & 3) != 0) {  // the founder sets the slot
                sk = make_float4(gt * kx.x, gt * kx.y, gt * kx.z, gt * kx.w);
                sv = make_float4(gt * vx.x, gt * vx.y, gt * vx.z, gt * vx.w);
                cnt = 1;
                rho = sqrtf(half_sum(dot4(vx, vx), hm));
            } else {
                sk = make_float4(fmaf(gt, kx.x, sk.x), fmaf(gt, kx.y, sk.y), fmaf(gt, kx.z, sk.z), fmaf(gt, kx.w, sk.w));
                sv = make_float4(fmaf(gt, vx.x, sv.x), fmaf(gt, vx.y, sv.y), fmaf(gt, vx.z, sv.z), fmaf(gt, vx.w, sv.w));
                ++cnt;
            }
        }
        // tokens that joined at this event are in every state from it on: pass 2 takes their
        // gradient as the total minus the sums before this event, kept here (the read-row
        // gradients of this event are already in registers)
        if (joined) {
            *reinterpret_cast<float4*>(a.dks + o) = Pk;
            *reinterpret_cast<float4*>(a.dvs + o) = Pv;
            if (hl == 0) a.drho[((int64_t)bh * a.E + e) * M + j] = Pr;
        }
        // read-row gradients -> sum and radius gradients of the state after event e
        const float cn = (float)(cnt > 0 ? cnt : 1);
        const float4 x = make_float4(sk.x / cn, sk.y / cn, sk.z / cn, sk.w / cn);
        const float mu = half_sum(sum4(x), hm) * (1.0f / D);
        const float4 xc = make_float4(x.x - mu, x.y - mu, x.z - mu, x.w - mu);
        const float var = half_sum(dot4(xc, xc), hm) * (1.0f / D);
        const float isd = 1.0f / sqrtf(var + a.ln_eps);
        const float4 xh = make_float4(xc.x * isd, xc.y * isd, xc.z * isd, xc.w * isd);
        // the rotary dims of the read key are constant zeros
        if (d0 < r) gkh.x = 0.0f;
        if (d0 + 1 < r) gkh.y = 0.0f;
        if (d0 + 2 < r) gkh.z = 0.0f;
        if (d0 + 3 < r) gkh.w = 0.0f;
        const float mg = half_sum(sum4(gkh), hm) * (1.0f / D);
        const float mgx = half_sum(dot4(gkh, xh), hm) * (1.0f / D);
        const float f = isd / cn;
        Pk = make_float4(Pk.x + (gkh.x - mg - xh.x * mgx) * f, Pk.y + (gkh.y - mg - xh.y * mgx) * f,
                         Pk.z + (gkh.z - mg - xh.z * mgx) * f, Pk.w + (gkh.w - mg - xh.w * mgx) * f);
        if (a.no_vnorm) {
            Pv = make_float4(Pv.x + gvh.x / cn, Pv.y + gvh.y / cn, Pv.z + gvh.z / cn, Pv.w + gvh.w / cn);
        } else {
            const float nv = sqrtf(half_sum(dot4(sv, sv), hm));
            const float inv = nv > 0.0f ? 1.0f / nv : 0.0f;
            const float4 u = make_float4(sv.x * inv, sv.y * inv, sv.z * inv, sv.w * inv);
            const float dr = half_sum(dot4(u, gvh), hm);
            const float fr = rho * inv;
            Pv = make_float4(Pv.x + fr * (gvh.x - u.x * dr), Pv.y + fr * (gvh.y - u.y * dr),
                             Pv.z + fr * (gvh.z - u.z * dr), Pv.w + fr * (gvh.w - u.w * dr));
            Pr += dr;
        }
    }
    // pass 2: member t joined at event t / C; its sum gradient is the slot's total over all
    // events minus the running sums kept at that event in pass 1
    for (int p = m0; p < m1; ++p) {
        const int ent = member(p, true);
        const int64_t t = ent >> 2;
        const int64_t eo = ((int64_t)bh * a.E + t / C) * M + j;
        const float4 bk = *reinterpret_cast<const float4*>(a.dks + eo * D + d0);
        const float4 bv = *reinterpret_cast<const float4*>(a.dvs + eo * D + d0);
        const float4 Gk = make_float4(Pk.x - bk.x, Pk.y - bk.y, Pk.z - bk.z, Pk.w - bk.w);
        const float4 Gv = make_float4(Pv.x - bv.x, Pv.y - bv.y, Pv.z - bv.z, Pv.w - bv.w);
        const float gt = gg[t];
        const float4 kx = ld4<T>(kk + t * D + d0), vx = ld4<T>(vv + t * D + d0);
        float4* dkp = reinterpret_cast<float4*>(a.dk + (row + t) * D + d0);
        float4* dvp = reinterpret_cast<float4*>(a.dv + (row + t) * D + d0);
        float4 dkt = *dkp, dvt = *dvp;
        dkt = make_float4(fmaf(gt, Gk.x, dkt.x), fmaf(gt, Gk.y, dkt.y), fmaf(gt, Gk.z, dkt.z), fmaf(gt, Gk.w, dkt.w));
        dvt = make_float4(fmaf(gt, Gv.x, dvt.x), fmaf(gt, Gv.y, dvt.y), fmaf(gt, Gv.z, dvt.z), fmaf(gt, Gv.w, dvt.w));
        if ((ent & 3) != 0) {  // founder: rho = |v|
            const float Gr = Pr - a.drho[eo];
            const float nv = sqrtf(half_sum(dot4(vx, vx), hm));
            const float fr = nv > 0.0f ? Gr / nv : 0.0f;
            dvt = make_float4(fmaf(fr, vx.x, dvt.x), fmaf(fr, vx.y, dvt.y), fmaf(fr, vx.z, dvt.z), fmaf(fr, vx.w, dvt.w));
        }
        *dkp = dkt;
        *dvp = dvt;
        const float dgt = half_sum(dot4(kx, Gk) + dot4(vx, Gv), hm);
        if (hl == 0) a.dg[row + t] += dgt;
    }
}

// ---------------------------------------------------------------- tiled path
// Chunks a multiple of 64: one CTA per (row, 64-query tile), 256 threads.  The tile's
// queries and dout stay in shared memory (row-major and transposed); its keys come in
// blocks of 64 (the read rows of its chunk's state, then its window), and per block the
// five products S = Q K^T, dP = dO V^T, dQ += dS K, dK = dS^T Q, dV = P^T dO run as
// 64 x 64 x 64 fp32 multiplies, each thread owning a 4 x 4 piece of every output.  A first
// pass over the blocks gives each query its log2-sum-exp.  dK and dV of a block are added
// to global accumulators (a window key is seen by W/C + 1 chunks; a read row by its one
// chunk's two tiles).
constexpr int TQ = 64, TKB = 64, TPAD = 68;  // tile rows, key-block rows, padded row (floats)
constexpr int TILE_SMEM = (10 * TQ * TPAD + 2 * TQ) * (int)sizeof(float);

template <typename T>
__device__ __forceinline__ void tile_load(float* rm, float* tr, const T* src, int nrows, int tid) {
    // rows [0, nrows) of src (64 dims each) into rm[r][x] and tr[x][r]; the rest zero
    for (int q = tid; q < TQ * (D / 4); q += 256) {
        const int r = q >> 4, x0 = (q & 15) * 4;
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        if (r < nrows) {
            if (sizeof(T) == 2) {
                const uint2 w = *reinterpret_cast<const uint2*>(src + (int64_t)r * D + x0);
                v[0] = __uint_as_float(w.x << 16);
                v[1] = __uint_as_float(w.x & 0xffff0000u);
                v[2] = __uint_as_float(w.y << 16);
                v[3] = __uint_as_float(w.y & 0xffff0000u);
            } else {
                const float4 f = *reinterpret_cast<const float4*>(src + (int64_t)r * D + x0);
                v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
            }
        }
        if (rm) *reinterpret_cast<float4*>(rm + r * TPAD + x0) = make_float4(v[0], v[1], v[2], v[3]);
        if (tr)
#pragma unroll
            for (int u = 0; u < 4; ++u) tr[(x0 + u) * TPAD + r] = v[u];
    }
}

// acc[4][4] += A^T-slab product: sum over k of a[k][i0..i0+3] * b[k][j0..j0+3]
__device__ __forceinline__ void mm4x4(float (&acc)[4][4], const float* a, const float* b, int i0, int j0, int K) {
#pragma unroll 8
    for (int k = 0; k < K; ++k) {
        const float4 x = *reinterpret_cast<const float4*>(a + k * TPAD + i0);
        const float4 y = *reinterpret_cast<const float4*>(b + k * TPAD + j0);
        const float xa[4] = {x.x, x.y, x.z, x.w}, ya[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(xa[i], ya[j], acc[i][j]);
    }
}

template <typename T>
__global__ void __launch_bounds__(256, 1) bwd_tile(BackwardArgs a) {
    extern __shared__ float tsm[];
    float* Qs = tsm;                 // [64][TPAD] rotated queries, row-major
    float* Qt = Qs + TQ * TPAD;      // transposed
    float* Gs = Qt + TQ * TPAD;      // dout, row-major
    float* Gt = Gs + TQ * TPAD;      // transposed
    float* Ks = Gt + TQ * TPAD;      // key block, row-major
    float* Kt = Ks + TQ * TPAD;      // transposed
    float* Vt = Kt + TQ * TPAD;      // value block, transposed
    float* Ps = Vt + TQ * TPAD;      // P, row-major [query][key]
    float* Ds = Ps + TQ * TPAD;      // dS, row-major
    float* Dt = Ds + TQ * TPAD;      // dS transposed [key][query]
    float* Ls = Dt + TQ * TPAD;      // log2-sum-exp per query
    float* Dd = Ls + TQ;             // dout . out per query
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const int i0 = 4 * ty, j0 = 4 * tx;
    const int tiles = (int)((a.N + TQ - 1) / TQ);
    const int bh = blockIdx.x / tiles;
    const int64_t q0 = (int64_t)(blockIdx.x % tiles) * TQ;
    const int nq = (int)(a.N - q0 < TQ ? a.N - q0 : TQ);
    const int Wc = a.W / a.C;
    const int64_t c = q0 / a.C, e = c - Wc - 1, ws = c - Wc > 0 ? (c - Wc) * a.C : 0;
    const int n = e >= 0 ? a.sched[e].n_after : 0;
    const int64_t row = (int64_t)bh * a.N;
    const int64_t plane = ((int64_t)bh * a.snap_events + (e >= 0 ? e : 0)) * a.M * D;
    const T* kh = reinterpret_cast<const T*>(a.snap_k) + plane;
    const T* vh = reinterpret_cast<const T*>(a.snap_v) + plane;
    const T* kr = reinterpret_cast<const T*>(a.kr) + row * D;
    const T* vv = reinterpret_cast<const T*>(a.v) + row * D;
    const int nbs = (n + TKB - 1) / TKB;
    const int nbw = (int)((q0 + nq - ws + TKB - 1) / TKB);
    const float sl = a.scale_log2;

    tile_load<T>(Qs, Qt, reinterpret_cast<const T*>(a.qr) + (row + q0) * D, nq, tid);
    tile_load<T>(Gs, Gt, reinterpret_cast<const T*>(a.dout) + (row + q0) * D, nq, tid);
    // dout . out of every query (four threads a row)
    {
        const int r = tid >> 2, part = tid & 3;
        float d = 0.0f;
        if (r < nq) {
            const T* o = reinterpret_cast<const T*>(a.out) + (row + q0 + r) * D + 16 * part;
            const T* g = reinterpret_cast<const T*>(a.dout) + (row + q0 + r) * D + 16 * part;
            for (int x = 0; x < 16; ++x) d = fmaf(to_f<T>(o[x]), to_f<T>(g[x]), d);
        }
        d += __shfl_xor_sync(0xffffffffu, d, 1);
        d += __shfl_xor_sync(0xffffffffu, d, 2);
        if (part == 0) Dd[r] = d;
    }
    // key block b: rows, values and the count of valid keys; window blocks mask causally
    auto load_block = [&](int b, bool want_v) -> int {
        int kv;
        if (b < nbs) {
            kv = n - TKB * b < TKB ? n - TKB * b : TKB;
            tile_load<T>(Ks, Kt, kh + (int64_t)TKB * b * D, kv, tid);
            if (want_v) tile_load<T>(nullptr, Vt, vh + (int64_t)TKB * b * D, kv, tid);
        } else {
            const int64_t t0 = ws + (int64_t)TKB * (b - nbs);
            kv = (int)(q0 + nq - t0 < TKB ? q0 + nq - t0 : TKB);
            tile_load<T>(Ks, Kt, kr + t0 * D, kv, tid);
            if (want_v) tile_load<T>(nullptr, Vt, vv + t0 * D, kv, tid);
        }
        return kv;
    };
    auto scores = [&](int b, int kv, float (&sc)[4][4]) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) sc[i][j] = 0.0f;
        mm4x4(sc, Qt, Kt, i0, j0, D);
        const bool win = b >= nbs;
        const int64_t t0 = win ? ws + (int64_t)TKB * (b - nbs) : 0;
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const bool ok = i0 + i < nq && j0 + j < kv && (!win || t0 + j0 + j <= q0 + i0 + i);
                sc[i][j] = ok ? sc[i][j] * sl : -INFINITY;
            }
    };
    // pass 1: log2-sum-exp of each query over all its keys
    float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY}, l[4] = {0.f, 0.f, 0.f, 0.f};
    for (int b = 0; b < nbs + nbw; ++b) {
        __syncthreads();
        const int kv = load_block(b, false);
        __syncthreads();
        float sc[4][4];
        scores(b, kv, sc);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float mb = fmaxf(fmaxf(sc[i][0], sc[i][1]), fmaxf(sc[i][2], sc[i][3]));
            const float mn = fmaxf(m[i], mb);
            if (mn == -INFINITY) continue;
            float add = 0.0f;
#pragma unroll
            for (int j = 0; j < 4; ++j) add += exp2f(sc[i][j] - mn);
            l[i] = l[i] * exp2f(m[i] - mn) + add;
            m[i] = mn;
        }
    }
    // combine the 16 threads of a row (a half-warp)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float M = m[i];
        for (int o = 8; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float L = m[i] == -INFINITY ? 0.0f : l[i] * exp2f(m[i] - M);
        for (int o = 8; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        if (tx == 0) Ls[i0 + i] = M + log2f(L);
    }
    // pass 2: the gradients
    float dq[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) dq[i][j] = 0.0f;
    for (int b = 0; b < nbs + nbw; ++b) {
        __syncthreads();
        const int kv = load_block(b, true);
        __syncthreads();
        float sc[4][4], dp[4][4];
        scores(b, kv, sc);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) dp[i][j] = 0.0f;
        mm4x4(dp, Gt, Vt, i0, j0, D);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float L = Ls[i0 + i], Dv = Dd[i0 + i];
            float pr[4], ds[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                pr[j] = sc[i][j] == -INFINITY ? 0.0f : exp2f(sc[i][j] - L);
                ds[j] = pr[j] * (dp[i][j] - Dv);
                Dt[(j0 + j) * TPAD + i0 + i] = ds[j];
            }
            *reinterpret_cast<float4*>(Ps + (i0 + i) * TPAD + j0) = make_float4(pr[0], pr[1], pr[2], pr[3]);
            *reinterpret_cast<float4*>(Ds + (i0 + i) * TPAD + j0) = make_float4(ds[0], ds[1], ds[2], ds[3]);
        }
        __syncthreads();
        // dQ += dS K (rows i0.., dims j0..)
        mm4x4(dq, Dt, Ks, i0, j0, TKB);
        // dK = dS^T Q and dV = P^T dO for keys 4ty.., dims 4tx.. (slabs over the queries)
        float dk[4][4], dv[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) dk[i][j] = dv[i][j] = 0.0f;
        mm4x4(dk, Ds, Qs, i0, j0, TQ);
        mm4x4(dv, Ps, Gs, i0, j0, TQ);
        const bool win = b >= nbs;
        const int64_t kbase = win ? ws + (int64_t)TKB * (b - nbs) : (int64_t)TKB * b;
        float* gk = win ? a.dk + (row + kbase) * D
                        : a.dks + (((int64_t)bh * a.E + e) * a.M + kbase) * D;
        float* gv = win ? a.dv + (row + kbase) * D
                        : a.dvs + (((int64_t)bh * a.E + e) * a.M + kbase) * D;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (i0 + i >= kv) continue;
            // four consecutive dims per vector atomic (16-byte aligned: j0 is a multiple of 4)
            const float s = a.inv_sqrt_d;
            atomicAdd(reinterpret_cast<float4*>(gk + (int64_t)(i0 + i) * D + j0),
                      make_float4(dk[i][0] * s, dk[i][1] * s, dk[i][2] * s, dk[i][3] * s));
            atomicAdd(reinterpret_cast<float4*>(gv + (int64_t)(i0 + i) * D + j0),
                      make_float4(dv[i][0], dv[i][1], dv[i][2], dv[i][3]));
        }
    }
    // dq: scaled, then rotated back (pairs across threads: through shared memory)
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float4*>(Ps + (i0 + i) * TPAD + j0) =
            make_float4(dq[i][0] * a.inv_sqrt_d, dq[i][1] * a.inv_sqrt_d, dq[i][2] * a.inv_sqrt_d, dq[i][3] * a.inv_sqrt_d);
    __syncthreads();
    const int half = a.r / 2;
    for (int q = tid; q < nq * D; q += 256) {
        const int r = q >> 6, x = q & 63;
        const int64_t pp = q0 + r;
        float y = Ps[r * TPAD + x];
        if (x < 2 * half) {
            const int i2 = x < half ? x : x - half;
            const float2 cs = a.rope[pp * half + i2];
            y = x < half ? y * cs.x + Ps[r * TPAD + x + half] * cs.y : y * cs.x - Ps[r * TPAD + x - half] * cs.y;
        }
        a.dq[(row + pp) * D + x] = y;
    }
}

// ------------------------------------------------------- tensor-core tiled path
// bf16 layers, chunks a multiple of 64: the same tiles as bwd_tile, the five products on
// the tensor cores (mma.sync m16n8k16, bf16 operands, fp32 accumulators; P and dS are
// rounded to bf16 for the three products that take them, as attention backwards do).
// Four warps; warp w owns query rows 16w .. 16w + 15 for S, dP and dQ, and keys
// 16w .. 16w + 15 of the block for dK and dV.  Operands come from padded shared-memory
// tiles by ldmatrix (transposed where a product needs the other major order).
constexpr int MQ = 64, MPAD = 72;  // tile rows; padded row of bf16 (144 bytes: conflict-free ldmatrix)

__device__ __forceinline__ uint32_t su32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ void ldm_x4(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(su32(p)));
}
__device__ __forceinline__ void ldm_x4_t(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(su32(p)));
}
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                 "{%0, %1, %2, %3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t packbf(float x, float y) {
    __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    return *reinterpret_cast<uint32_t*>(&h);
}

// rows [0, nrows) of a [., 64] bf16 array into a padded tile (zeros beyond)
__device__ __forceinline__ void mtile_load(__nv_bfloat16* t, const __nv_bfloat16* src, int nrows, int tid) {
    for (int q = tid; q < MQ * 8; q += 128) {
        const int r = q >> 3, c8 = (q & 7) * 8;
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (r < nrows) w = *reinterpret_cast<const uint4*>(src + (int64_t)r * D + c8);
        *reinterpret_cast<uint4*>(t + r * MPAD + c8) = w;
    }
}

// rows [0, nrows) of a [., 64] bf16 array into a padded tile by asynchronous copies
// (rows past nrows are zero-filled: a copy of 0 source bytes)
__device__ __forceinline__ void mtile_load_async(__nv_bfloat16* t, const __nv_bfloat16* src, int nrows, int tid) {
    for (int q = tid; q < MQ * 8; q += 128) {
        const int r = q >> 3, c8 = (q & 7) * 8;
        const bool ok = r < nrows;
        const __nv_bfloat16* g = ok ? src + (int64_t)r * D + c8 : src;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(su32(t + r * MPAD + c8)), "l"(g),
                     "r"(ok ? 16 : 0)
                     : "memory");
    }
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// acc[8 n-tiles] (16 rows x 64 cols) += A (16 x 64, rows a_row0.. of a row-major tile)
// times B^T where B is a row-major [n][k] tile (n = the 64 output columns)
__device__ __forceinline__ void mm_rows_nk(float (&acc)[8][4], const __nv_bfloat16* A, const __nv_bfloat16* B,
                                           int lane) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        uint32_t a[4];
        ldm_x4(a, A + (lane & 15) * MPAD + kk * 16 + (lane >> 4) * 8);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
            uint32_t b[4];  // n-tiles 2np, 2np + 1; k halves
            ldm_x4(b, B + (np * 16 + (lane & 7) + ((lane >> 4) << 3)) * MPAD + kk * 16 + ((lane >> 3) & 1) * 8);
            mma16816(acc[2 * np], a, b[0], b[1]);
            mma16816(acc[2 * np + 1], a, b[2], b[3]);
        }
    }
}
// acc (16 x 64 dims) += A (16 x 64 along k, from registers) times B where B is a
// row-major [k][n] tile
__device__ __forceinline__ void mm_regs_kn(float (&acc)[8][4], const uint32_t (&a)[4][4], const __nv_bfloat16* B,
                                           int lane) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
        for (int np = 0; np < 4; ++np) {
            uint32_t b[4];
            ldm_x4_t(b, B + (kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * MPAD + np * 16 + (lane >> 4) * 8);
            mma16816(acc[2 * np], a[kk], b[0], b[1]);
            mma16816(acc[2 * np + 1], a[kk], b[2], b[3]);
        }
    }
}
// acc (16 keys x 64 dims) += A^T (A a row-major [k = query][m = key] tile, keys m0..)
// times B (a row-major [k = query][n = dim] tile)
__device__ __forceinline__ void mm_tt(float (&acc)[8][4], const __nv_bfloat16* A, int m0, const __nv_bfloat16* B,
                                      int lane) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        uint32_t a[4];
        ldm_x4_t(a, A + (kk * 16 + (lane & 7) + (lane >> 4) * 8) * MPAD + m0 + ((lane >> 3) & 1) * 8);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
            uint32_t b[4];
            ldm_x4_t(b, B + (kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * MPAD + np * 16 + (lane >> 4) * 8);
            mma16816(acc[2 * np], a, b[0], b[1]);
            mma16816(acc[2 * np + 1], a, b[2], b[3]);
        }
    }
}

constexpr int MTILE_SMEM = 8 * MQ * MPAD * 2 + 2 * MQ * 4;

__global__ void __launch_bounds__(128) bwd_tile_tc(BackwardArgs a) {
    extern __shared__ __align__(16) uint8_t msm[];
    __nv_bfloat16* Qs = reinterpret_cast<__nv_bfloat16*>(msm);
    __nv_bfloat16* Gs = Qs + MQ * MPAD;   // dout
    __nv_bfloat16* Ks = Gs + MQ * MPAD;
    __nv_bfloat16* Vs = Ks + MQ * MPAD;
    __nv_bfloat16* Ps = Vs + MQ * MPAD;   // P [query][key]
    __nv_bfloat16* Ss = Ps + MQ * MPAD;   // dS [query][key]
    __nv_bfloat16* K2 = Ss + MQ * MPAD;   // second K / V buffers (the next block's copies)
    __nv_bfloat16* V2 = K2 + MQ * MPAD;
    float* Ls = reinterpret_cast<float*>(V2 + MQ * MPAD);
    float* Dd = Ls + MQ;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t4 = lane & 3;
    const int tiles = (int)((a.N + MQ - 1) / MQ);
    const int bh = blockIdx.x / tiles;
    const int64_t q0 = (int64_t)(blockIdx.x % tiles) * MQ;
    const int nq = (int)(a.N - q0 < MQ ? a.N - q0 : MQ);
    const int Wc = a.W / a.C;
    const int64_t c = q0 / a.C, e = c - Wc - 1, ws = c - Wc > 0 ? (c - Wc) * a.C : 0;
    const int n = e >= 0 ? a.sched[e].n_after : 0;
    const int64_t row = (int64_t)bh * a.N;
    const int64_t plane = ((int64_t)bh * a.snap_events + (e >= 0 ? e : 0)) * a.M * D;
    const __nv_bfloat16* kh = reinterpret_cast<const __nv_bfloat16*>(a.snap_k) + plane;
    const __nv_bfloat16* vh = reinterpret_cast<const __nv_bfloat16*>(a.snap_v) + plane;
    const __nv_bfloat16* kr = reinterpret_cast<const __nv_bfloat16*>(a.kr) + row * D;
    const __nv_bfloat16* vv = reinterpret_cast<const __nv_bfloat16*>(a.v) + row * D;
    const int nbs = (n + MQ - 1) / MQ;
    const int nbw = (int)((q0 + nq - ws + MQ - 1) / MQ);
    const float sl = a.scale_log2;
    const int r0 = 16 * warp;  // this warp's query rows (and keys of a block for dK, dV)

    mtile_load(Qs, reinterpret_cast<const __nv_bfloat16*>(a.qr) + (row + q0) * D, nq, tid);
    mtile_load(Gs, reinterpret_cast<const __nv_bfloat16*>(a.dout) + (row + q0) * D, nq, tid);
    {   // dout . out per query (two threads a row)
        const int r = tid >> 1, part = tid & 1;
        float d = 0.0f;
        if (r < nq) {
            const __nv_bfloat16* o = reinterpret_cast<const __nv_bfloat16*>(a.out) + (row + q0 + r) * D + 32 * part;
            const __nv_bfloat16* gp = reinterpret_cast<const __nv_bfloat16*>(a.dout) + (row + q0 + r) * D + 32 * part;
            for (int x = 0; x < 32; ++x) d = fmaf(__bfloat162float(o[x]), __bfloat162float(gp[x]), d);
        }
        d += __shfl_xor_sync(0xffffffffu, d, 1);
        if (part == 0) Dd[r] = d;
    }
    auto load_block = [&](int b, bool want_v) -> int {
        int kv;
        if (b < nbs) {
            kv = n - MQ * b < MQ ? n - MQ * b : MQ;
            mtile_load(Ks, kh + (int64_t)MQ * b * D, kv, tid);
            if (want_v) mtile_load(Vs, vh + (int64_t)MQ * b * D, kv, tid);
        } else {
            const int64_t t0 = ws + (int64_t)MQ * (b - nbs);
            kv = (int)(q0 + nq - t0 < MQ ? q0 + nq - t0 : MQ);
            mtile_load(Ks, kr + t0 * D, kv, tid);
            if (want_v) mtile_load(Vs, vv + t0 * D, kv, tid);
        }
        return kv;
    };
    // scores of this warp's rows (fragment rows g, g + 8; columns 8 nt + 2 t4, + 1), log2 units
    auto scores = [&](int b, int kv, const __nv_bfloat16* Kb, float (&sc)[8][4]) {
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int u = 0; u < 4; ++u) sc[nt][u] = 0.0f;
        mm_rows_nk(sc, Qs + r0 * MPAD, Kb, lane);
        const bool win = b >= nbs;
        const int64_t t0 = win ? ws + (int64_t)MQ * (b - nbs) : 0;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int qi = r0 + g + (u >> 1) * 8, kj = nt * 8 + 2 * t4 + (u & 1);
                const bool ok = qi < nq && kj < kv && (!win || t0 + kj <= q0 + qi);
                sc[nt][u] = ok ? sc[nt][u] * sl : -INFINITY;
            }
    };
    // pass 1: log2-sum-exp per query (the forward's, when it kept them)
    float m2[2] = {-INFINITY, -INFINITY}, l2[2] = {0.f, 0.f};
    if (a.lse_fwd) {
        for (int rr = tid; rr < MQ; rr += 128) Ls[rr] = rr < nq ? a.lse_fwd[row + q0 + rr] : 0.0f;
        __syncthreads();
    }
    for (int b = 0; a.lse_fwd == nullptr && b < nbs + nbw; ++b) {
        __syncthreads();
        const int kv = load_block(b, false);
        __syncthreads();
        float sc[8][4];
        scores(b, kv, Ks, sc);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float mb = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) mb = fmaxf(mb, fmaxf(sc[nt][2 * h], sc[nt][2 * h + 1]));
            const float mn = fmaxf(m2[h], mb);
            if (mn == -INFINITY) continue;
            float add = 0.0f;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) add += exp2f(sc[nt][2 * h] - mn) + exp2f(sc[nt][2 * h + 1] - mn);
            l2[h] = l2[h] * exp2f(m2[h] - mn) + add;
            m2[h] = mn;
        }
    }
#pragma unroll
    for (int h = 0; h < 2 && a.lse_fwd == nullptr; ++h) {  // the four threads of a row
        float M = m2[h];
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 1));
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 2));
        float L = m2[h] == -INFINITY ? 0.0f : l2[h] * exp2f(m2[h] - M);
        L += __shfl_xor_sync(0xffffffffu, L, 1);
        L += __shfl_xor_sync(0xffffffffu, L, 2);
        if (t4 == 0) Ls[r0 + g + 8 * h] = M + log2f(L);
    }
    __syncwarp();
    // pass 2
    float dq[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
        for (int u = 0; u < 4; ++u) dq[nt][u] = 0.0f;
    // K and V blocks double-buffered: block b + 1 is copied while block b is worked on
    auto block_rows = [&](int b) -> int {
        if (b < nbs) return n - MQ * b < MQ ? n - MQ * b : MQ;
        const int64_t t0 = ws + (int64_t)MQ * (b - nbs);
        return (int)(q0 + nq - t0 < MQ ? q0 + nq - t0 : MQ);
    };
    auto issue_block = [&](int b, __nv_bfloat16* kd, __nv_bfloat16* vd) {
        const int kv = block_rows(b);
        if (b < nbs) {
            mtile_load_async(kd, kh + (int64_t)MQ * b * D, kv, tid);
            mtile_load_async(vd, vh + (int64_t)MQ * b * D, kv, tid);
        } else {
            const int64_t t0 = ws + (int64_t)MQ * (b - nbs);
            mtile_load_async(kd, kr + t0 * D, kv, tid);
            mtile_load_async(vd, vv + t0 * D, kv, tid);
        }
        cp_async_commit();
    };
    const int nblocks = nbs + nbw;
    __syncthreads();  // pass 1 is done with the K buffer
    issue_block(0, Ks, Vs);
    for (int b = 0; b < nblocks; ++b) {
        __nv_bfloat16* Kc = (b & 1) ? K2 : Ks;
        __nv_bfloat16* Vc = (b & 1) ? V2 : Vs;
        // the other buffers were last read by block b - 1's S, dP and dQ products, which
        // every thread finished before block b - 1's barrier ahead of its dK, dV products
        if (b + 1 < nblocks) {
            issue_block(b + 1, (b & 1) ? Ks : K2, (b & 1) ? Vs : V2);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();  // every thread's copies of block b have landed
        const int kv = block_rows(b);
        float sc[8][4], dp[8][4];
        scores(b, kv, Kc, sc);
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int u = 0; u < 4; ++u) dp[nt][u] = 0.0f;
        mm_rows_nk(dp, Gs + r0 * MPAD, Vc, lane);
        uint32_t afrag[4][4];  // dS as A fragments (keys along k) for dQ
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int qi = r0 + g + 8 * h;
            const float L = Ls[qi], Dv = Dd[qi];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const float p0 = sc[nt][2 * h] == -INFINITY ? 0.0f : exp2f(sc[nt][2 * h] - L);
                const float p1 = sc[nt][2 * h + 1] == -INFINITY ? 0.0f : exp2f(sc[nt][2 * h + 1] - L);
                const float d0 = p0 * (dp[nt][2 * h] - Dv), d1 = p1 * (dp[nt][2 * h + 1] - Dv);
                const uint32_t pp = packbf(p0, p1), dd = packbf(d0, d1);
                *reinterpret_cast<uint32_t*>(Ps + qi * MPAD + nt * 8 + 2 * t4) = pp;
                *reinterpret_cast<uint32_t*>(Ss + qi * MPAD + nt * 8 + 2 * t4) = dd;
                // A fragment of k-step nt/2: regs 0/1 (rows g / g+8) from the even n-tile,
                // 2/3 from the odd one
                afrag[nt >> 1][(nt & 1) * 2 + h] = dd;
            }
        }
        // dQ += dS K
        mm_regs_kn(dq, afrag, Kc, lane);
        __syncthreads();  // P and dS of every warp are in shared memory
        // dK = dS^T Q, dV = P^T dO for keys r0 .. r0 + 15 of the block
        float dk[8][4], dv[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int u = 0; u < 4; ++u) dk[nt][u] = dv[nt][u] = 0.0f;
        mm_tt(dk, Ss, r0, Qs, lane);
        mm_tt(dv, Ps, r0, Gs, lane);
        const bool win = b >= nbs;
        const int64_t kbase = win ? ws + (int64_t)MQ * (b - nbs) : (int64_t)MQ * b;
        float* gk = win ? a.dk + (row + kbase) * D : a.dks + (((int64_t)bh * a.E + e) * a.M + kbase) * D;
        float* gv = win ? a.dv + (row + kbase) * D : a.dvs + (((int64_t)bh * a.E + e) * a.M + kbase) * D;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int kj = r0 + g + 8 * h;
            if (kj >= kv) continue;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                const int dd0 = nt * 8 + 2 * t4;
                // two consecutive dims per vector atomic (8-byte aligned: dd0 is even)
                atomicAdd(reinterpret_cast<float2*>(gk + (int64_t)kj * D + dd0),
                          make_float2(dk[nt][2 * h] * a.inv_sqrt_d, dk[nt][2 * h + 1] * a.inv_sqrt_d));
                atomicAdd(reinterpret_cast<float2*>(gv + (int64_t)kj * D + dd0),
                          make_float2(dv[nt][2 * h], dv[nt][2 * h + 1]));
            }
        }
    }
    // dq: scaled and rotated back (pairs across threads: through shared memory as fp32)
    __syncthreads();
    float* Fq = reinterpret_cast<float*>(msm);  // [64][64] fp32 over the Q / dout tiles
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const int qi = r0 + g + 8 * h, x = nt * 8 + 2 * t4;
            Fq[qi * D + x] = dq[nt][2 * h] * a.inv_sqrt_d;
            Fq[qi * D + x + 1] = dq[nt][2 * h + 1] * a.inv_sqrt_d;
        }
    __syncthreads();
    const int half = a.r / 2;
    for (int q = tid; q < nq * D; q += 128) {
        const int rr = q >> 6, x = q & 63;
        const int64_t pp = q0 + rr;
        float y = Fq[rr * D + x];
        if (x < 2 * half) {
            const int i2 = x < half ? x : x - half;
            const float2 cs = a.rope[pp * half + i2];
            y = x < half ? y * cs.x + Fq[rr * D + x + half] * cs.y : y * cs.x - Fq[rr * D + x - half] * cs.y;
        }
        a.dq[(row + pp) * D + x] = y;
    }
}

// rotate the accumulated window-key gradients back (in place) and zero the gate gradient
__global__ void bwd_unrotate_dk(BackwardArgs a) {
    const int64_t rows = (int64_t)a.BH * a.N;
    const int half = a.r / 2;
    for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < rows * half;
         w += (int64_t)gridDim.x * blockDim.x) {
        const int64_t rr = w / half;
        const int i = (int)(w - rr * half);
        const int64_t p = rr % a.N;
        float* k = a.dk + rr * D;
        const float2 cs = a.rope[p * half + i];
        const float y0 = k[i], y1 = k[i + half];
        k[i] = y0 * cs.x + y1 * cs.y;
        k[i + half] = y1 * cs.x - y0 * cs.y;
    }
}

template <typename T>
cudaError_t launch_all(const BackwardArgs& a, cudaStream_t s) {
    const int64_t rows = (int64_t)a.BH * a.N;
    if (rows == 0) return cudaSuccess;
    const int wpb = BW_WARPS;
    const unsigned gq = (unsigned)((rows + wpb - 1) / wpb);
    bwd_rotate<T><<<2048, 256, 0, s>>>(a);
    if (a.C % TQ == 0) {
        // tiled path: gradients accumulate into zeroed outputs and read-row arrays
        cudaError_t e = cudaMemsetAsync(a.dk, 0, (size_t)rows * D * sizeof(float), s);
        if (e == cudaSuccess) e = cudaMemsetAsync(a.dv, 0, (size_t)rows * D * sizeof(float), s);
        if (e == cudaSuccess) e = cudaMemsetAsync(a.dg, 0, (size_t)rows * sizeof(float), s);
        const size_t rs = (size_t)a.BH * a.E * a.M * D * sizeof(float);
        const bool tc5 = sizeof(T) == 2 && bwd_tc5_supported(a, true);
        const bool zero_rows = !(tc5 && bwd_tc5_owns_read_rows(a));
        if (e == cudaSuccess && a.E > 0 && zero_rows) e = cudaMemsetAsync(a.dks, 0, rs, s);
        if (e == cudaSuccess && a.E > 0 && zero_rows) e = cudaMemsetAsync(a.dvs, 0, rs, s);
        if (e != cudaSuccess) return e;
        static bool attr = false;
        if (!attr) {
            cudaFuncSetAttribute(bwd_tile<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, TILE_SMEM);
            cudaFuncSetAttribute(bwd_tile_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, MTILE_SMEM);
            attr = true;
        }
        const int tiles = (int)((a.N + TQ - 1) / TQ);
        if (tc5) {
            e = launch_bwd_tc5(a, s);
            if (e != cudaSuccess) return e;
        } else if (sizeof(T) == 2) {
            bwd_tile_tc<<<(unsigned)(a.BH * tiles), 128, MTILE_SMEM, s>>>(a);
        } else {
            bwd_tile<T><<<(unsigned)(a.BH * tiles), 256, TILE_SMEM, s>>>(a);
        }
        if (a.r > 0) bwd_unrotate_dk<<<2048, 256, 0, s>>>(a);
    } else {
        bwd_stats<T><<<gq, BW_THREADS, 0, s>>>(a);
        bwd_dq<T><<<gq, BW_THREADS, 0, s>>>(a);
        bwd_dkv_win<T><<<gq, BW_THREADS, 0, s>>>(a);
        if (a.E > 0) {
            const int64_t ws = (int64_t)a.BH * a.E * a.M;
            bwd_dstate<T><<<(unsigned)((ws + wpb - 1) / wpb), BW_THREADS, 0, s>>>(a);
        }
    }
    if (a.E > 0) {
        const int64_t slots = (int64_t)a.BH * a.M;
        bwd_members<<<(unsigned)a.BH, MB_THREADS, (size_t)(a.M + 1 + MB_STAGE) * sizeof(int), s>>>(a);
        // two slots a warp
        bwd_sweep16<T><<<(unsigned)(((slots + 1) / 2 + SW_WARPS - 1) / SW_WARPS), SW_WARPS * 32, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward(const BackwardArgs& a, bool bf16, cudaStream_t s) {
    if (a.C > MAX_BW_C) return cudaErrorInvalidValue;
    return bf16 ? launch_all<__nv_bfloat16>(a, s) : launch_all<float>(a, s);
}

}  // namespace kvm
