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
// Kernels (fp32 arithmetic, inputs in the layer's dtype; one warp per query,
// key or state row, lanes over the 64 dims, two each):
//   bwd_rotate   q and k rotated at their own positions (scratch)
//   bwd_stats    per query: log2-sum-exp of its scores and D = dout . out
//   bwd_dq       per query: dq (state part in plain coordinates, window part
//                rotated back)
//   bwd_dkv_win  per key: dk (rotated back) and dv from the queries whose
//                window holds it; dgate = 0
//   bwd_dstate   per fold event and slot: the gradient of the event's read
//                rows (key and value) from the chunk that reads them
//   bwd_sweep    per (batch, head) row, one CTA: replays the fold with the
//                recorded decisions (the forward's fp32 sums, in its order),
//                turns each event's read-row gradients into sum and radius
//                gradients (LayerNorm and normalisation backward), and sums
//                them from the last event back to each token's own event,
//                adding the tokens' k, v and gate gradients.
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

template <typename T>
__global__ void __launch_bounds__(BW_THREADS) bwd_sweep(BackwardArgs a) {
    __shared__ int slot[MAX_BW_C], kd[MAX_BW_C], ord[MAX_BW_C], run_beg[MAX_BW_C + 1];
    __shared__ int nruns_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int bh = blockIdx.x;
    const int C = a.C, M = a.M;
    const int64_t row = (int64_t)bh * a.N;
    const T* kk = reinterpret_cast<const T*>(a.k) + row * D;
    const T* vv = reinterpret_cast<const T*>(a.v) + row * D;
    const float* gg = a.g + row;
    float* sk = a.sk + (int64_t)bh * M * D;
    float* sv = a.sv + (int64_t)bh * M * D;
    int* cnt = a.cnt + (int64_t)bh * M;
    float* rho = a.rho + (int64_t)bh * M;
    float* gk = a.gk + (int64_t)bh * M * D;
    float* gv = a.gv + (int64_t)bh * M * D;
    float* grho = a.grho + (int64_t)bh * M;
    const int r = a.r;

    // an entry of the record that names no slot of this state, or no kind, is
    // reported and its token skipped (kind -1)
    auto load_event = [&](int e) {
        const int n = a.sched[e].n_after;
        for (int i = tid; i < C; i += BW_THREADS) {
            const int64_t o = ((int64_t)bh * a.rec_events + e) * C + i;
            const int j = a.assign[o], kn = a.kind[o];
            const bool ok = j >= 0 && j < n && kn >= 0 && kn <= 2;
            if (!ok && a.status) atomicOr(a.status, STATUS_DEVICE);
            slot[i] = ok ? j : 0;
            kd[i] = ok ? kn : -1;
        }
    };
    for (int i = tid; i < M * D; i += BW_THREADS) {
        sk[i] = 0.0f;
        sv[i] = 0.0f;
    }
    for (int i = tid; i < M; i += BW_THREADS) {
        cnt[i] = 1;  // a slot merged into before any founding (an invalid record) divides by 1
        rho[i] = 0.0f;
    }
    __syncthreads();

    // pass 1: replay the fold; each event's read-row gradients become sum / radius gradients
    for (int e = 0; e < a.E; ++e) {
        load_event(e);
        __syncthreads();
        // founders: the new slot's sums, count 1, radius |v|
        for (int i = warp; i < C; i += BW_WARPS) {
            if (kd[i] != 1 && kd[i] != 2) continue;
            const int j = slot[i];
            const int64_t t = (int64_t)e * C + i;
            const float gt = gg[t];
            const float2 kx = ld2<T>(kk + t * D + 2 * lane), vx = ld2<T>(vv + t * D + 2 * lane);
            reinterpret_cast<float2*>(sk + (int64_t)j * D)[lane] = make_float2(gt * kx.x, gt * kx.y);
            reinterpret_cast<float2*>(sv + (int64_t)j * D)[lane] = make_float2(gt * vx.x, gt * vx.y);
            const float nv = sqrtf(warp_sum(dot2(vx, vx)));
            if (lane == 0) {
                cnt[j] = 1;
                rho[j] = nv;
            }
        }
        // merged tokens sorted by (slot, position): runs of one slot, in position order
        if (tid < C) {
            int rank = 0;
            if (kd[tid] == 0) {
                const int si = slot[tid];
                for (int u = 0; u < C; ++u)
                    rank += kd[u] == 0 && (slot[u] < si || (slot[u] == si && u < tid));
                ord[rank] = tid;
            }
        }
        const int nm = __syncthreads_count(tid < C && kd[tid] == 0);
        if (tid == 0) {
            int nr = 0;
            for (int q = 0; q < nm; ++q)
                if (q == 0 || slot[ord[q]] != slot[ord[q - 1]]) run_beg[nr++] = q;
            run_beg[nr] = nm;
            nruns_s = nr;
        }
        __syncthreads();
        for (int ru = warp; ru < nruns_s; ru += BW_WARPS) {
            const int j = slot[ord[run_beg[ru]]];
            float2 xk = reinterpret_cast<const float2*>(sk + (int64_t)j * D)[lane];
            float2 xv = reinterpret_cast<const float2*>(sv + (int64_t)j * D)[lane];
            for (int q = run_beg[ru]; q < run_beg[ru + 1]; ++q) {
                const int64_t t = (int64_t)e * C + ord[q];
                const float gt = gg[t];
                const float2 kx = ld2<T>(kk + t * D + 2 * lane), vx = ld2<T>(vv + t * D + 2 * lane);
                xk = make_float2(fmaf(gt, kx.x, xk.x), fmaf(gt, kx.y, xk.y));
                xv = make_float2(fmaf(gt, vx.x, xv.x), fmaf(gt, vx.y, xv.y));
            }
            reinterpret_cast<float2*>(sk + (int64_t)j * D)[lane] = xk;
            reinterpret_cast<float2*>(sv + (int64_t)j * D)[lane] = xv;
            if (lane == 0) cnt[j] += run_beg[ru + 1] - run_beg[ru];
        }
        __syncthreads();
        // read-row gradients -> sum and radius gradients of the state after event e
        const int n = a.sched[e].n_after;
        for (int j = warp; j < n; j += BW_WARPS) {
            const int64_t o = (((int64_t)bh * a.E + e) * M + j) * D;
            const float cn = (float)cnt[j];
            const float2 s = reinterpret_cast<const float2*>(sk + (int64_t)j * D)[lane];
            const float2 x = make_float2(s.x / cn, s.y / cn);
            const float mu = warp_sum(x.x + x.y) * (1.0f / D);
            const float2 xc = make_float2(x.x - mu, x.y - mu);
            const float var = warp_sum(dot2(xc, xc)) * (1.0f / D);
            const float isd = 1.0f / sqrtf(var + a.ln_eps);
            const float2 xh = make_float2(xc.x * isd, xc.y * isd);
            float2 gkh = reinterpret_cast<const float2*>(a.dks + o)[lane];
            if (2 * lane < r) gkh.x = 0.0f;  // the rotary dims of the read key are constant zeros
            if (2 * lane + 1 < r) gkh.y = 0.0f;
            const float mg = warp_sum(gkh.x + gkh.y) * (1.0f / D);
            const float mgx = warp_sum(dot2(gkh, xh)) * (1.0f / D);
            const float2 dsk = make_float2((gkh.x - mg - xh.x * mgx) * isd / cn, (gkh.y - mg - xh.y * mgx) * isd / cn);
            const float2 gvh = reinterpret_cast<const float2*>(a.dvs + o)[lane];
            const float2 svv = reinterpret_cast<const float2*>(sv + (int64_t)j * D)[lane];
            float2 dsv;
            float dr = 0.0f;
            if (a.no_vnorm) {
                dsv = make_float2(gvh.x / cn, gvh.y / cn);
            } else {
                const float nv = sqrtf(warp_sum(dot2(svv, svv)));
                const float inv = nv > 0.0f ? 1.0f / nv : 0.0f;
                const float2 u = make_float2(svv.x * inv, svv.y * inv);
                dr = warp_sum(dot2(u, gvh));
                const float f = rho[j] * inv;
                dsv = make_float2(f * (gvh.x - u.x * dr), f * (gvh.y - u.y * dr));
            }
            reinterpret_cast<float2*>(a.dks + o)[lane] = dsk;
            reinterpret_cast<float2*>(a.dvs + o)[lane] = dsv;
            if (lane == 0) a.drho[((int64_t)bh * a.E + e) * M + j] = dr;
        }
        __syncthreads();
    }

    // pass 2: from the last event back, G = sum of the gradients of every state that
    // holds a token's contribution; each token reads G at its own event
    for (int i = tid; i < M * D; i += BW_THREADS) {
        gk[i] = 0.0f;
        gv[i] = 0.0f;
    }
    for (int i = tid; i < M; i += BW_THREADS) grho[i] = 0.0f;
    __syncthreads();
    for (int e = a.E - 1; e >= 0; --e) {
        load_event(e);
        const int n = a.sched[e].n_after;
        const int64_t base = ((int64_t)bh * a.E + e) * M;
        for (int i = tid; i < n * D; i += BW_THREADS) {
            gk[i] += a.dks[base * D + i];
            gv[i] += a.dvs[base * D + i];
        }
        for (int i = tid; i < n; i += BW_THREADS) grho[i] += a.drho[base + i];
        __syncthreads();
        for (int i = warp; i < C; i += BW_WARPS) {
            const int kdi = kd[i];
            if (kdi < 0) continue;
            const int j = slot[i];
            const int64_t t = (int64_t)e * C + i;
            const float gt = gg[t];
            const float2 kx = ld2<T>(kk + t * D + 2 * lane), vx = ld2<T>(vv + t * D + 2 * lane);
            const float2 Gk = reinterpret_cast<const float2*>(gk + (int64_t)j * D)[lane];
            const float2 Gv = reinterpret_cast<const float2*>(gv + (int64_t)j * D)[lane];
            float2* dkp = reinterpret_cast<float2*>(a.dk + (row + t) * D) + lane;
            float2* dvp = reinterpret_cast<float2*>(a.dv + (row + t) * D) + lane;
            float2 dk = *dkp, dv = *dvp;
            dk.x = fmaf(gt, Gk.x, dk.x);
            dk.y = fmaf(gt, Gk.y, dk.y);
            dv.x = fmaf(gt, Gv.x, dv.x);
            dv.y = fmaf(gt, Gv.y, dv.y);
            if (kdi == 1 || kdi == 2) {  // founder: rho = |v|
                const float nv = sqrtf(warp_sum(dot2(vx, vx)));
                const float f = nv > 0.0f ? grho[j] / nv : 0.0f;
                dv.x = fmaf(f, vx.x, dv.x);
                dv.y = fmaf(f, vx.y, dv.y);
            }
            *dkp = dk;
            *dvp = dv;
            const float dgt = warp_sum(dot2(kx, Gk) + dot2(vx, Gv));
            if (lane == 0) a.dg[row + t] += dgt;
        }
        __syncthreads();
    }
}

template <typename T>
cudaError_t launch_all(const BackwardArgs& a, cudaStream_t s) {
    const int64_t rows = (int64_t)a.BH * a.N;
    if (rows == 0) return cudaSuccess;
    const int wpb = BW_WARPS;
    const unsigned gq = (unsigned)((rows + wpb - 1) / wpb);
    bwd_rotate<T><<<2048, 256, 0, s>>>(a);
    bwd_stats<T><<<gq, BW_THREADS, 0, s>>>(a);
    bwd_dq<T><<<gq, BW_THREADS, 0, s>>>(a);
    bwd_dkv_win<T><<<gq, BW_THREADS, 0, s>>>(a);
    if (a.E > 0) {
        const int64_t ws = (int64_t)a.BH * a.E * a.M;
        bwd_dstate<T><<<(unsigned)((ws + wpb - 1) / wpb), BW_THREADS, 0, s>>>(a);
        bwd_sweep<T><<<a.BH, BW_THREADS, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward(const BackwardArgs& a, bool bf16, cudaStream_t s) {
    if (a.C > MAX_BW_C) return cudaErrorInvalidValue;
    return bf16 ? launch_all<__nv_bfloat16>(a, s) : launch_all<float>(a, s);
}

}  // namespace kvm
