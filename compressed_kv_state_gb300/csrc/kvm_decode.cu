// KVM decode step: one new token per (batch, head).
//
// "Key-Value Means" (gist.science technical summary), Problem statement
// (decode cost of plain attention grows with the context) and Core
// mechanisms 1 and 4; chatpaper.ai abstract ("long context decoding").
// The new token's unrotated key, value and gate enter the window ring, then
// its query attends, in one softmax, to the state's read view (unrotated
// query) and to window tokens (c - W/C)*C .. p (RoPE on both sides).  A fold
// at a chunk boundary runs before this kernel (fold chain, one event).
#include "kvm_internal.cuh"

namespace kvm {

constexpr int DEC_THREADS = 128;

template <typename T>
__global__ void __launch_bounds__(DEC_THREADS) decode_kernel(DecodeArgs a) {
    __shared__ float qs[D];
    __shared__ float kbuf[DEC_THREADS / 32][D];
    __shared__ float accs[DEC_THREADS / 32][D];
    __shared__ float ls[DEC_THREADS / 32], mxs[DEC_THREADS / 32];
    const int bh = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int L = a.W + a.C;
    const int64_t p = a.pos;
    const int half = a.r / 2;
    T* rk = reinterpret_cast<T*>(a.ring_k) + (int64_t)bh * L * D;
    T* rv = reinterpret_cast<T*>(a.ring_v) + (int64_t)bh * L * D;

    // the new token enters the ring
    if (tid < D) {
        const int64_t sl = (p % L) * D + tid;
        rk[sl] = reinterpret_cast<const T*>(a.k)[(int64_t)bh * D + tid];
        rv[sl] = reinterpret_cast<const T*>(a.v)[(int64_t)bh * D + tid];
    }
    if (tid == 0) a.ring_g[(int64_t)bh * L + p % L] = a.g[bh];
    // rotated, scaled query
    if (tid < D) {
        const T* q = reinterpret_cast<const T*>(a.q) + (int64_t)bh * D;
        float x = to_f<T>(q[tid]);
        if (tid < 2 * half) {
            const int i = tid < half ? tid : tid - half;
            const float2 cs = a.rope[p * half + i];
            x = tid < half ? x * cs.x - to_f<T>(q[tid + half]) * cs.y
                           : x * cs.x + to_f<T>(q[tid - half]) * cs.y;
        }
        qs[tid] = x * a.scale_log2;
    }
    __syncthreads();

    const int64_t c = p / a.C, Wc = a.W / a.C;
    const int64_t ws = c - Wc > 0 ? (c - Wc) * a.C : 0;
    const int n = a.n_slots;
    const int64_t nkeys = n + (p - ws + 1);
    const T* vk = reinterpret_cast<const T*>(a.view_k) + (int64_t)bh * a.M * D;
    const T* vv = reinterpret_cast<const T*>(a.view_v) + (int64_t)bh * a.M * D;

    // each warp takes keys warp, warp + 4, ...; lanes split the head dim (2 each)
    float m = -INFINITY, l = 0.0f, acc0 = 0.0f, acc1 = 0.0f;
    const float q0 = qs[lane], q1 = qs[lane + 32];
    for (int64_t j = warp; j < nkeys; j += DEC_THREADS / 32) {
        float k0, k1, v0, v1;
        if (j < n) {
            k0 = to_f<T>(vk[j * D + lane]);
            k1 = to_f<T>(vk[j * D + lane + 32]);
            v0 = to_f<T>(vv[j * D + lane]);
            v1 = to_f<T>(vv[j * D + lane + 32]);
        } else {
            const int64_t kp = ws + (j - n);
            const int64_t sl = (kp % L) * D;
            k0 = to_f<T>(rk[sl + lane]);
            k1 = to_f<T>(rk[sl + lane + 32]);
            if (half > 0) {
                // rotate-half RoPE at the key's own position: pair (i, i + half)
                kbuf[warp][lane] = k0;
                kbuf[warp][lane + 32] = k1;
                __syncwarp();
                const float2* rp = a.rope + kp * half;
                if (lane < half) {
                    const float2 cs = rp[lane];
                    k0 = kbuf[warp][lane] * cs.x - kbuf[warp][lane + half] * cs.y;
                } else if (lane < 2 * half) {
                    const float2 cs = rp[lane - half];
                    k0 = kbuf[warp][lane] * cs.x + kbuf[warp][lane - half] * cs.y;
                }
                const int x1 = lane + 32;
                if (x1 < half) {
                    const float2 cs = rp[x1];
                    k1 = kbuf[warp][x1] * cs.x - kbuf[warp][x1 + half] * cs.y;
                } else if (x1 < 2 * half) {
                    const float2 cs = rp[x1 - half];
                    k1 = kbuf[warp][x1] * cs.x + kbuf[warp][x1 - half] * cs.y;
                }
                __syncwarp();
            }
            v0 = to_f<T>(rv[sl + lane]);
            v1 = to_f<T>(rv[sl + lane + 32]);
        }
        const float s = warp_sum(q0 * k0 + q1 * k1);
        const float mnew = fmaxf(m, s);
        const float corr = exp2f(m - mnew);
        const float pj = exp2f(s - mnew);
        l = l * corr + pj;
        acc0 = acc0 * corr + pj * v0;
        acc1 = acc1 * corr + pj * v1;
        m = mnew;
    }
    if (lane == 0) {
        mxs[warp] = m;
        ls[warp] = l;
    }
    accs[warp][lane] = acc0;
    accs[warp][lane + 32] = acc1;
    __syncthreads();
    if (tid < D) {
        float M = -INFINITY;
        for (int w = 0; w < DEC_THREADS / 32; ++w) M = fmaxf(M, mxs[w]);
        float L2 = 0.0f, o = 0.0f;
        for (int w = 0; w < DEC_THREADS / 32; ++w) {
            const float f = mxs[w] == -INFINITY ? 0.0f : exp2f(mxs[w] - M);
            L2 += ls[w] * f;
            o += accs[w][tid] * f;
        }
        reinterpret_cast<T*>(a.out)[(int64_t)bh * D + tid] = from_f<T>(o / L2);
    }
}

cudaError_t launch_decode(const DecodeArgs& a, bool bf16, cudaStream_t s) {
    if (bf16)
        decode_kernel<__nv_bfloat16><<<a.BH, DEC_THREADS, 0, s>>>(a);
    else
        decode_kernel<float><<<a.BH, DEC_THREADS, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kvm
