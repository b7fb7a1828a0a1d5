// Portable KVM attention for the prefill: one query per thread, fp32 math.
//
// "Key-Value Means" (gist.science technical summary), Methodology and Core
// mechanism 4: one softmax over the compressed state (state keys zero on the
// rotary dims, read by the unrotated query) and the block-sliding window
// (RoPE on query and keys).  Query p of chunk c sees the state as it stands
// after chunk c - W/C - 1 was folded and the window tokens (c - W/C)*C .. p.
//
// This kernel serves the fp32 dtype and every shape the tensor-core kernel
// does not cover.  Because the key view is exactly zero on dims [0, r), the
// rotated query gives the same state scores as the unrotated one, so one
// rotated query register file serves both parts.
#include "kvm_internal.cuh"

namespace kvm {

constexpr int KT = 32;  // keys per shared-memory tile

template <typename T>
__global__ void __launch_bounds__(64) attn_simt_kernel(AttnArgs a, int QB) {
    __shared__ float ks[KT][D];
    __shared__ float vs[KT][D];
    const int bh = blockIdx.y;
    const int tid = threadIdx.x;
    const int64_t p0 = (int64_t)blockIdx.x * QB;
    const int64_t p = p0 + tid;
    const bool valid = p < a.N;
    const int64_t c = p0 / a.C;
    const int64_t Wc = a.W / a.C;
    const int64_t e = c - Wc - 1;  // last event folded before chunk c
    const int n = e >= 0 ? a.sched[e].n_after : 0;
    const int64_t ws = c - Wc > 0 ? (c - Wc) * a.C : 0;
    const int64_t kend = min(a.N, p0 + QB);
    const int half = a.r / 2;

    const T* qrow = reinterpret_cast<const T*>(a.q) + ((int64_t)bh * a.N + (valid ? p : p0)) * D;
    const T* kb = reinterpret_cast<const T*>(a.k) + (int64_t)bh * a.N * D;
    const T* vb = reinterpret_cast<const T*>(a.v) + (int64_t)bh * a.N * D;

    float qr[D];
#pragma unroll
    for (int x = 0; x < D; ++x) qr[x] = to_f<T>(qrow[x]);
    {
        const float2* rp = a.rope + (valid ? p : p0) * half;
#pragma unroll
        for (int i = 0; i < D / 2; ++i) {
            if (i < half) {
                const float2 cs = rp[i];
                const float x0 = qr[i], x1 = qr[i + half];
                qr[i] = x0 * cs.x - x1 * cs.y;
                qr[i + half] = x1 * cs.x + x0 * cs.y;
            }
        }
    }
#pragma unroll
    for (int x = 0; x < D; ++x) qr[x] *= a.scale_log2;

    float m = -INFINITY, l = 0.0f;
    float acc[D];
#pragma unroll
    for (int x = 0; x < D; ++x) acc[x] = 0.0f;

    auto process = [&](int cnt, int64_t key_pos0, bool causal) {
        float s[KT];
        float tmax = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < KT; ++jj) {
            float d = 0.0f;
#pragma unroll
            for (int x = 0; x < D; ++x) d = fmaf(qr[x], ks[jj][x], d);
            const bool ok = jj < cnt && (!causal || key_pos0 + jj <= p);
            s[jj] = ok ? d : -INFINITY;
            tmax = fmaxf(tmax, s[jj]);
        }
        if (tmax == -INFINITY) return;
        const float mnew = fmaxf(m, tmax);
        const float corr = exp2f(m - mnew);
        l *= corr;
#pragma unroll
        for (int x = 0; x < D; ++x) acc[x] *= corr;
#pragma unroll
        for (int jj = 0; jj < KT; ++jj) {
            const float pj = exp2f(s[jj] - mnew);
            l += pj;
#pragma unroll
            for (int x = 0; x < D; ++x) acc[x] = fmaf(pj, vs[jj][x], acc[x]);
        }
        m = mnew;
    };

    // state rows (snapshot after event e)
    if (n > 0) {
        const T* sk = reinterpret_cast<const T*>(a.snap_k) + ((int64_t)bh * a.snap_events + e) * a.M * D;
        const T* sv = reinterpret_cast<const T*>(a.snap_v) + ((int64_t)bh * a.snap_events + e) * a.M * D;
        for (int j0 = 0; j0 < n; j0 += KT) {
            const int cnt = min(KT, n - j0);
            __syncthreads();
            for (int i = tid; i < KT * D; i += blockDim.x) {
                const int jj = i / D, x = i % D;
                ks[jj][x] = jj < cnt ? to_f<T>(sk[(int64_t)(j0 + jj) * D + x]) : 0.0f;
                vs[jj][x] = jj < cnt ? to_f<T>(sv[(int64_t)(j0 + jj) * D + x]) : 0.0f;
            }
            __syncthreads();
            process(cnt, 0, false);
        }
    }
    // window keys with RoPE at their own positions, causal
    for (int64_t k0 = ws; k0 < kend; k0 += KT) {
        const int cnt = (int)min((int64_t)KT, kend - k0);
        __syncthreads();
        for (int i = tid; i < KT * D; i += blockDim.x) {
            const int jj = i / D, x = i % D;
            float kv = 0.0f, vv = 0.0f;
            if (jj < cnt) {
                const int64_t kp = k0 + jj;
                const T* kr = kb + kp * D;
                kv = to_f<T>(kr[x]);
                if (x < 2 * half) {
                    const int i2 = x < half ? x : x - half;
                    const float2 cs = a.rope[kp * half + i2];
                    if (x < half)
                        kv = kv * cs.x - to_f<T>(kr[x + half]) * cs.y;
                    else
                        kv = kv * cs.x + to_f<T>(kr[x - half]) * cs.y;
                }
                vv = to_f<T>(vb[kp * D + x]);
            }
            ks[jj][x] = kv;
            vs[jj][x] = vv;
        }
        __syncthreads();
        process(cnt, k0, true);
    }

    if (valid) {
        T* orow = reinterpret_cast<T*>(a.out) + ((int64_t)bh * a.N + p) * D;
        const float il = 1.0f / l;
#pragma unroll
        for (int x = 0; x < D; ++x) orow[x] = from_f<T>(acc[x] * il);
    }
}

// Window ring: tokens [first, N) of each row enter the ring (row = position mod L)
// with their unrotated key (for folds and export), value, gate, and a copy of the
// key rotated at the token's position (for decode attention).  rotate_only:
// rebuild only the rotated copy from the ring's own keys.
template <typename T>
__global__ void ring_fill_kernel(RingFillArgs a) {
    const int bh = blockIdx.y;
    const int half = a.r / 2;
    const int64_t cnt = a.N - a.first;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < cnt * D;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t tok = a.first + i / D;
        const int x = (int)(i % D);
        const int64_t slot = tok % a.L;
        const int64_t dst = ((int64_t)bh * a.L + slot) * D + x;
        const T* krow;
        if (a.rotate_only) {
            krow = reinterpret_cast<const T*>(a.ring_k) + ((int64_t)bh * a.L + slot) * D;
        } else {
            const int64_t src = ((int64_t)bh * a.N + tok) * D;
            krow = reinterpret_cast<const T*>(a.k) + src;
            reinterpret_cast<T*>(a.ring_k)[dst] = krow[x];
            reinterpret_cast<T*>(a.ring_v)[dst] = reinterpret_cast<const T*>(a.v)[src + x];
            if (x == 0) a.ring_g[(int64_t)bh * a.L + slot] = a.g[(int64_t)bh * a.N + tok];
        }
        float kv = to_f<T>(krow[x]);
        if (x < 2 * half) {
            const int i2 = x < half ? x : x - half;
            const float2 cs = a.rope[tok * half + i2];
            kv = x < half ? kv * cs.x - to_f<T>(krow[x + half]) * cs.y : kv * cs.x + to_f<T>(krow[x - half]) * cs.y;
        }
        reinterpret_cast<T*>(a.ring_kr)[dst] = from_f<T>(kv);
    }
}

// One thread per 16-byte chunk (8 dims) of a key row: chunks inside the rotary
// dims are rotated with their rotate-half partner chunk (vector path when r/2
// is a multiple of 8, one dim at a time otherwise); the rest are copied.  Rows
// (b, h) are strided over gridDim.y and chunks of a row over gridDim.x, so the
// position of a chunk needs no division.
// Rotate the 16-byte chunk c (dims 8c .. 8c+7) of row p of src (row-major [N][8] chunks)
// in place in w: rotate-half pairs (x, x + half) on the rotary dims [0, r).
__device__ __forceinline__ void rope_chunk(const uint4* src, int64_t p, int c, int r, const float2* rope, uint4& w) {
    const int half = r / 2;
    if (8 * c >= r) return;
    if ((half & 7) == 0) {
        const int hc = half >> 3;
        const bool low = c < hc;  // dims [0, half) pair with [half, r)
        const uint4 o = src[p * 8 + (low ? c + hc : c - hc)];
        const float4* tab = reinterpret_cast<const float4*>(rope + p * half + (low ? c : c - hc) * 8);
        const float4 t[4] = {tab[0], tab[1], tab[2], tab[3]};
        const float ce[8] = {t[0].x, t[0].z, t[1].x, t[1].z, t[2].x, t[2].z, t[3].x, t[3].z};
        const float se[8] = {t[0].y, t[0].w, t[1].y, t[1].w, t[2].y, t[2].w, t[3].y, t[3].w};
        __nv_bfloat162* m2 = reinterpret_cast<__nv_bfloat162*>(&w);
        const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&o);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float2 mv = __bfloat1622float2(m2[u]), ov = __bfloat1622float2(o2[u]);
            const float c0 = ce[2 * u], c1 = ce[2 * u + 1], s0 = se[2 * u], s1 = se[2 * u + 1];
            m2[u] = low ? __floats2bfloat162_rn(mv.x * c0 - ov.x * s0, mv.y * c1 - ov.y * s1)
                        : __floats2bfloat162_rn(mv.x * c0 + ov.x * s0, mv.y * c1 + ov.y * s1);
        }
    } else {
        const __nv_bfloat16* krow = reinterpret_cast<const __nv_bfloat16*>(src + p * 8);
        __nv_bfloat16* m = reinterpret_cast<__nv_bfloat16*>(&w);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int x = 8 * c + e;
            if (x < 2 * half) {
                const int i2 = x < half ? x : x - half;
                const float2 cs = rope[p * half + i2];
                const float kv = __bfloat162float(krow[x]);
                const float r2 = x < half ? kv * cs.x - __bfloat162float(krow[x + half]) * cs.y
                                          : kv * cs.x + __bfloat162float(krow[x - half]) * cs.y;
                m[e] = __float2bfloat16_rn(r2);
            }
        }
    }
}

// The loads a rotated 16-byte piece of a key and of a query needs (each piece, its
// rotate-half partner, and their shared (cos, sin) entries) are issued before any
// arithmetic (the vector path: r/2 a multiple of 8).
__device__ __forceinline__ uint4 rope_apply(uint4 w, const uint4& o, const float4 (&t)[4], bool low) {
    const float ce[8] = {t[0].x, t[0].z, t[1].x, t[1].z, t[2].x, t[2].z, t[3].x, t[3].z};
    const float se[8] = {t[0].y, t[0].w, t[1].y, t[1].w, t[2].y, t[2].w, t[3].y, t[3].w};
    __nv_bfloat162* m2 = reinterpret_cast<__nv_bfloat162*>(&w);
    const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&o);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const float2 mv = __bfloat1622float2(m2[u]), ov = __bfloat1622float2(o2[u]);
        const float c0 = ce[2 * u], c1 = ce[2 * u + 1], s0 = se[2 * u], s1 = se[2 * u + 1];
        m2[u] = low ? __floats2bfloat162_rn(mv.x * c0 - ov.x * s0, mv.y * c1 - ov.y * s1)
                    : __floats2bfloat162_rn(mv.x * c0 + ov.x * s0, mv.y * c1 + ov.y * s1);
    }
    return w;
}

// One thread per 16-byte piece (8 dims) of a row.  Full rows: every piece of k and q is
// written to k_rot / q_rot (the rotary pieces rotated).  Compact rows: only the r / 8
// rotary pieces are (rows of r dims).  Ring tokens get their whole rows in the ring.
// Compact rows: the ring tokens' pieces past the rotary dims (pieces RC .. 7), as they are.
__device__ __forceinline__ void ring_rest_compact(const RopeKeysArgs& a, int bh, int RC) {
    const int64_t row0 = (int64_t)bh * a.N * 8;
    const uint4* src = reinterpret_cast<const uint4*>(a.k) + row0;
    const int NR = 8 - RC;
    const int64_t cnt = (a.N - a.first) * NR;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < cnt; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t p = a.first + i / NR;
        const int c = RC + (int)(i % NR);
        const int64_t fi = p * 8 + c;
        const int64_t slot = p - (p / a.L) * a.L;
        const int64_t rrow = (int64_t)bh * a.L + slot;
        const uint4 w = src[fi];
        reinterpret_cast<uint4*>(a.ring_k)[rrow * 8 + c] = w;
        reinterpret_cast<uint4*>(a.ring_v)[rrow * 8 + c] = reinterpret_cast<const uint4*>(a.v)[row0 + fi];
        reinterpret_cast<uint4*>(a.ring_kr)[rrow * 8 + c] = w;
    }
}

// Compact rows, r = 32: one thread per rotate-half pair of pieces (u, u + 2) of a
// position: the two pieces of k and q and their shared (cos, sin) entries are loaded
// once for both outputs.
__device__ __forceinline__ void rope_pairs_compact(const RopeKeysArgs& a) {
    constexpr int RC = 4, HC = 2;  // pieces of a compact row; pairs per position
    const int half = 16;
    const int64_t items = a.N * HC;
    for (int bh = blockIdx.y; bh < a.BH; bh += gridDim.y) {
        const int64_t row0 = (int64_t)bh * a.N * 8;
        const uint4* src = reinterpret_cast<const uint4*>(a.k) + row0;
        const uint4* qsrc = reinterpret_cast<const uint4*>(a.q) + row0;
        uint4* dst = reinterpret_cast<uint4*>(a.k_rot) + (int64_t)bh * a.N * RC;
        uint4* qdst = reinterpret_cast<uint4*>(a.q_rot) + (int64_t)bh * a.N * RC;
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < items;
             i += (int64_t)gridDim.x * blockDim.x) {
            const int64_t p = i >> 1;
            const int u = (int)(i & 1);
            const uint4 klo = src[p * 8 + u], khi = src[p * 8 + u + HC];
            const uint4 qlo = qsrc[p * 8 + u], qhi = qsrc[p * 8 + u + HC];
            const float4* tab = reinterpret_cast<const float4*>(a.rope + p * half + u * 8);
            const float4 t[4] = {tab[0], tab[1], tab[2], tab[3]};
            const uint4 rlo = rope_apply(klo, khi, t, true), rhi = rope_apply(khi, klo, t, false);
            dst[p * RC + u] = rlo;
            dst[p * RC + u + HC] = rhi;
            qdst[p * RC + u] = rope_apply(qlo, qhi, t, true);
            qdst[p * RC + u + HC] = rope_apply(qhi, qlo, t, false);
            if (a.ring_k && p >= a.first) {  // the window ring: whole rows (the rest below)
                const int64_t slot = p - (p / a.L) * a.L;
                const int64_t rrow = (int64_t)bh * a.L + slot;
                const uint4* vs = reinterpret_cast<const uint4*>(a.v) + row0;
                uint4* rk = reinterpret_cast<uint4*>(a.ring_k) + rrow * 8;
                uint4* rv = reinterpret_cast<uint4*>(a.ring_v) + rrow * 8;
                uint4* rkr = reinterpret_cast<uint4*>(a.ring_kr) + rrow * 8;
                rk[u] = klo;
                rk[u + HC] = khi;
                rv[u] = vs[p * 8 + u];
                rv[u + HC] = vs[p * 8 + u + HC];
                rkr[u] = rlo;
                rkr[u + HC] = rhi;
                if (u == 0) a.ring_g[rrow] = a.g[(int64_t)bh * a.N + p];
            }
        }
        if (a.ring_k) ring_rest_compact(a, bh, RC);
    }
}

__global__ void rope_keys_kernel(RopeKeysArgs a) {
    if (a.compact && a.q) {
        rope_pairs_compact(a);
        return;
    }
    const int RC = a.compact ? a.r / 8 : 8;  // pieces of a k_rot / q_rot row
    const int lg = RC == 8 ? 3 : (RC == 4 ? 2 : (RC == 2 ? 1 : 0));
    const int64_t per_row = a.N * RC;
    const int half = a.r / 2, hc = half >> 3;
    const bool vec = (half & 7) == 0;
    for (int bh = blockIdx.y; bh < a.BH; bh += gridDim.y) {
        const int64_t row0 = (int64_t)bh * a.N * 8;  // first piece of this row in k, q, v
        const uint4* src = reinterpret_cast<const uint4*>(a.k) + row0;
        uint4* dst = reinterpret_cast<uint4*>(a.k_rot) + (int64_t)bh * per_row;
        const uint4* qsrc = a.q ? reinterpret_cast<const uint4*>(a.q) + row0 : nullptr;
        uint4* qdst = a.q ? reinterpret_cast<uint4*>(a.q_rot) + (int64_t)bh * per_row : nullptr;
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < per_row;
             i += (int64_t)gridDim.x * blockDim.x) {
            const int64_t p = i >> lg;
            const int c = (int)(i & (RC - 1));
            const int64_t fi = p * 8 + c;  // the piece in a full row
            const bool rot = 8 * c < a.r, low = c < hc;
            const int64_t partner = p * 8 + (low ? c + hc : c - hc);
            // every load of this piece first
            uint4 w = src[fi], wq = make_uint4(0u, 0u, 0u, 0u), o = w, oq = w;
            float4 t[4];
            if (qsrc) wq = qsrc[fi];
            if (vec && rot) {
                o = src[partner];
                if (qsrc) oq = qsrc[partner];
                const float4* tab = reinterpret_cast<const float4*>(a.rope + p * half + (low ? c : c - hc) * 8);
#pragma unroll
                for (int u = 0; u < 4; ++u) t[u] = tab[u];
            }
            const bool ring = a.ring_k && p >= a.first;
            int64_t rrow = 0;
            if (ring) {
                const int64_t slot = p - (p / a.L) * a.L;
                rrow = (int64_t)bh * a.L + slot;
                reinterpret_cast<uint4*>(a.ring_k)[rrow * 8 + c] = w;
                reinterpret_cast<uint4*>(a.ring_v)[rrow * 8 + c] = reinterpret_cast<const uint4*>(a.v)[row0 + fi];
                if (c == 0) a.ring_g[rrow] = a.g[(int64_t)bh * a.N + p];
            }
            if (vec) {
                if (rot) {
                    w = rope_apply(w, o, t, low);
                    if (qsrc) wq = rope_apply(wq, oq, t, low);
                }
            } else {
                rope_chunk(src, p, c, a.r, a.rope, w);
                if (qsrc) rope_chunk(qsrc, p, c, a.r, a.rope, wq);
            }
            dst[i] = w;
            if (ring) reinterpret_cast<uint4*>(a.ring_kr)[rrow * 8 + c] = w;
            if (qsrc) qdst[i] = wq;
        }
        // compact rows: the ring tokens' pieces past the rotary dims, as they are
        if (RC < 8 && a.ring_k) ring_rest_compact(a, bh, RC);
    }
}

cudaError_t launch_rope_keys(const RopeKeysArgs& a, cudaStream_t s) {
    if (a.N <= 0 || a.r <= 0) return cudaSuccess;
    // a.grid CTAs in total, spread over rows (y) and the chunks of a row (x)
    const int gy = a.BH < 65535 ? a.BH : 65535;
    int gx = a.grid / gy;
    if (a.compact && a.r != 32) return cudaErrorInvalidValue;
    const int64_t need = (a.N * (a.compact ? (a.q ? 2 : a.r / 8) : 8) + 255) / 256;
    if (gx < 1) gx = 1;
    if (gx > need) gx = (int)need;
    rope_keys_kernel<<<dim3((unsigned)gx, (unsigned)gy), 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_attn(const AttnArgs& a, bool bf16, cudaStream_t s) {
    if (a.N == 0) return cudaSuccess;
    if (attn_tc_supported(a, bf16)) return launch_attn_tc(a, a.status, s);
    const int QB = (a.C % 64 == 0) ? 64 : (a.C % 32 == 0 ? 32 : 16);
    dim3 grid((unsigned)((a.N + QB - 1) / QB), (unsigned)a.BH);
    if (bf16)
        attn_simt_kernel<__nv_bfloat16><<<grid, QB, 0, s>>>(a, QB);
    else
        attn_simt_kernel<float><<<grid, QB, 0, s>>>(a, QB);
    return cudaGetLastError();
}

cudaError_t launch_ring_fill(const RingFillArgs& a, bool bf16, cudaStream_t s) {
    const int64_t cnt = (a.N - a.first) * D;
    if (cnt <= 0) return cudaSuccess;
    const int64_t nb = (cnt + 255) / 256;
    dim3 grid((unsigned)(nb < 64 ? nb : 64), (unsigned)a.BH);
    if (bf16)
        ring_fill_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(a);
    else
        ring_fill_kernel<float><<<grid, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kvm
