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

constexpr int DEC_WARPS = 3;
constexpr int DEC_THREADS = DEC_WARPS * 32;
constexpr int TK = 32;  // keys per tile

__device__ __forceinline__ uint32_t dsmem_u32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

// bulk global -> shared copy completing on an mbarrier (16-byte aligned, multiple of 16 bytes)
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

template <typename T> __device__ __forceinline__ float2 ld2s(const T* p);
template <> __device__ __forceinline__ float2 ld2s<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(p));
}
template <> __device__ __forceinline__ float2 ld2s<float>(const float* p) { return *reinterpret_cast<const float2*>(p); }

// One CTA per (b, h), three warps (48 KB of stages: four CTAs per SM, so the
// 1024 rows of the decode sweep take two waves).  Keys (state rows, then the window in
// position order) are split into one contiguous range per warp; each warp
// streams its range in tiles of 32 keys through two shared-memory stages of
// its own, filled by bulk copies (a tile holds state rows only, or window rows
// only: the state's compact key rows (the non-rotary dims), or at most two
// contiguous runs of the window ring).
// Scores are dim-parallel (lane = 2 dims) with a butterfly transpose-reduce
// that leaves key i's score on lane i; P V is dim-parallel from shared memory;
// online softmax per warp, warps combined at the end.
template <typename T>
__global__ void __launch_bounds__(DEC_THREADS, 4) decode_kernel(DecodeArgs a) {
    constexpr int RB = 64 * (int)sizeof(T);  // bytes per key row
    constexpr int TILE = TK * RB;            // bytes of one K (or V) tile
    extern __shared__ __align__(128) uint8_t dsm[];
    __shared__ float qs[D];
    __shared__ float red_m[DEC_WARPS], red_l[DEC_WARPS];
    __shared__ float red_acc[DEC_WARPS][D];
    __shared__ __align__(8) unsigned long long bars[DEC_WARPS][2];
    const int bh = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int L = a.W + a.C;
    const int64_t p = a.pos;
    const int half = a.r / 2;
    T* rk = reinterpret_cast<T*>(a.ring_k) + (int64_t)bh * L * D;
    T* rv = reinterpret_cast<T*>(a.ring_v) + (int64_t)bh * L * D;
    T* rkr = reinterpret_cast<T*>(a.ring_kr) + (int64_t)bh * L * D;

    // the new token enters the rings (its key also rotated at position p); rotated, scaled query
    if (tid < D) {
        const int x = tid;
        const T* k = reinterpret_cast<const T*>(a.k) + (int64_t)bh * D;
        const T* q = reinterpret_cast<const T*>(a.q) + (int64_t)bh * D;
        const int64_t sl = (p % L) * D + x;
        rk[sl] = k[x];
        rv[sl] = reinterpret_cast<const T*>(a.v)[(int64_t)bh * D + x];
        float kx = to_f<T>(k[x]), qx = to_f<T>(q[x]);
        if (x < 2 * half) {
            const int i = x < half ? x : x - half;
            const float2 cs = a.rope[p * half + i];
            if (x < half) {
                kx = kx * cs.x - to_f<T>(k[x + half]) * cs.y;
                qx = qx * cs.x - to_f<T>(q[x + half]) * cs.y;
            } else {
                kx = kx * cs.x + to_f<T>(k[x - half]) * cs.y;
                qx = qx * cs.x + to_f<T>(q[x - half]) * cs.y;
            }
        }
        rkr[sl] = from_f<T>(kx);
        qs[x] = qx * a.scale_log2;
    }
    if (tid == 0) a.ring_g[(int64_t)bh * L + p % L] = a.g[bh];
    if (lane == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(dsmem_u32(&bars[warp][0])) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(dsmem_u32(&bars[warp][1])) : "memory");
    }
    // the bulk copies below read the rows just written through the generic proxy
    asm volatile("fence.proxy.async;" ::: "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();

    const int64_t c = p / a.C, Wc = a.W / a.C;
    const int64_t ws = c - Wc > 0 ? (c - Wc) * a.C : 0;
    const int ws_slot = (int)(ws % L);
    const int n = kvm_check(a.n_slots <= a.M, a.status) ? a.n_slots : 0;
    const int nkeys = n + (int)(p - ws + 1);
    // compact read-key rows: dims [D - DK, D) (the state keys are zero on the rotary dims)
    const int DK = view_k_dims(a.r), k0d = D - DK;
    const uint32_t RBK = (uint32_t)(DK * (int)sizeof(T));
    const T* vk = reinterpret_cast<const T*>(a.view_k) + (int64_t)bh * a.M * DK;
    const T* vv = reinterpret_cast<const T*>(a.view_v) + (int64_t)bh * a.M * D;
    const int per = ((nkeys + DEC_WARPS * TK - 1) / (DEC_WARPS * TK)) * TK;
    const int beg = warp * per, end = min(nkeys, beg + per);
    uint8_t* stage = dsm + warp * 2 * 2 * TILE;  // [2 stages][K tile, V tile]

    // a tile ends after TK keys, at the range's end, or where the state rows end
    auto tile_end = [&](int k0) {
        const int k1 = min(end, k0 + TK);
        return (k0 < n && k1 > n) ? n : k1;
    };
    // issue the copies of keys [k0, k1) into stage b (lane 0 only)
    auto issue = [&](int k0, int k1, int b) {
        const uint32_t bar = dsmem_u32(&bars[warp][b]);
        const uint32_t sk = dsmem_u32(stage + b * 2 * TILE), sv = sk + TILE;
        const bool st = k0 < n;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar),
                     "r"((uint32_t)(k1 - k0) * ((st ? RBK : (uint32_t)RB) + (uint32_t)RB)) : "memory");
        int kk = k0;
        if (st) {  // state rows (compact keys)
            bulk_g2s(sk, vk + (int64_t)kk * DK, (uint32_t)(k1 - kk) * RBK, bar);
            bulk_g2s(sv, vv + (int64_t)kk * D, (uint32_t)((k1 - kk) * RB), bar);
            kk = k1;
        }
        while (kk < k1) {  // window rows, contiguous up to the ring's end
            int slot = ws_slot + (kk - n);
            if (slot >= L) slot -= L;
            const int e = min(k1, kk + (L - slot));
            const uint32_t o = (uint32_t)((kk - k0) * RB);
            bulk_g2s(sk + o, rkr + (int64_t)slot * D, (uint32_t)((e - kk) * RB), bar);
            bulk_g2s(sv + o, rv + (int64_t)slot * D, (uint32_t)((e - kk) * RB), bar);
            kk = e;
        }
    };

    float m = -INFINITY, l = 0.0f, acc0 = 0.0f, acc1 = 0.0f;
    const float2 qv = make_float2(qs[2 * lane], qs[2 * lane + 1]);
    int it = 0;
    if (lane == 0 && beg < end) issue(beg, tile_end(beg), 0);
    __syncwarp();
    for (int k0 = beg, k1; k0 < end; k0 = k1, ++it) {
        const int b = it & 1;
        k1 = tile_end(k0);
        const int cnt = k1 - k0;
        if (lane == 0 && k1 < end) issue(k1, tile_end(k1), b ^ 1);
        // wait for this tile: every lane waits on the stage's barrier (try_wait suspends
        // the warp in hardware; bounded: a copy that never lands latches a timeout)
        {
            const uint32_t bar = dsmem_u32(&bars[warp][b]);
            const uint32_t par = (it >> 1) & 1;
            uint32_t ok = 0;
            long long t0 = -1;
            for (;;) {
                asm volatile("{\n\t.reg .pred q;\n\tmbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2;\n\tselp.u32 %0, 1, 0, q;\n\t}\n"
                             : "=r"(ok) : "r"(bar), "r"(par) : "memory");
                if (ok) break;
                if (t0 < 0) t0 = clock64();
                if (clock64() - t0 > (1ll << 32)) {
                    if (lane == 0 && a.status) atomicOr(a.status, STATUS_TIMEOUT);
                    break;
                }
            }
            if (!__all_sync(0xffffffffu, ok)) break;
        }
        const T* kt = reinterpret_cast<const T*>(stage + b * 2 * TILE);
        const T* vt = reinterpret_cast<const T*>(stage + b * 2 * TILE + TILE);
        // partial dot products of this lane's two dims with every key of the tile
        // (state rows: compact, nothing stored below dim D - DK; rows past cnt are
        // stale and masked after the reduction)
        float v[TK];
        if (k0 < n) {
            const bool has = 2 * lane >= k0d;
            const T* kl = kt + (has ? 2 * lane - k0d : 0);
#pragma unroll
            for (int j = 0; j < TK; ++j) {
                const float2 kx = has ? ld2s<T>(kl + j * DK) : make_float2(0.0f, 0.0f);
                v[j] = qv.x * kx.x + qv.y * kx.y;
            }
        } else {
#pragma unroll
            for (int j = 0; j < TK; ++j) {
                const float2 kx = ld2s<T>(kt + j * D + 2 * lane);
                v[j] = qv.x * kx.x + qv.y * kx.y;
            }
        }
        // butterfly transpose-reduce: afterwards lane i holds key i's score
#pragma unroll
        for (int off = 16, w = TK; off >= 1; off >>= 1, w >>= 1) {
            const bool upper = (lane & off) != 0;
#pragma unroll
            for (int i = 0; i < w / 2; ++i) {
                const float send = upper ? v[i] : v[i + w / 2];
                const float keep = upper ? v[i + w / 2] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
            }
        }
        const float sc = lane < cnt ? v[0] : -INFINITY;
        const float mnew = fmaxf(m, warp_max(sc));
        const float corr = exp2f(m - mnew);
        const float pj = exp2f(sc - mnew);
        l = l * corr + warp_sum(pj);
        acc0 *= corr;
        acc1 *= corr;
        m = mnew;
        if (cnt == TK) {
#pragma unroll
            for (int j = 0; j < TK; ++j) {
                const float pk = __shfl_sync(0xffffffffu, pj, j);
                const float2 vx = ld2s<T>(vt + j * D + 2 * lane);
                acc0 = fmaf(pk, vx.x, acc0);
                acc1 = fmaf(pk, vx.y, acc1);
            }
        } else {
#pragma unroll
            for (int j = 0; j < TK; ++j) {
                const float pk = __shfl_sync(0xffffffffu, pj, j);  // 0 past the tile's keys
                if (j < cnt) {
                    const float2 vx = ld2s<T>(vt + j * D + 2 * lane);
                    acc0 = fmaf(pk, vx.x, acc0);
                    acc1 = fmaf(pk, vx.y, acc1);
                }
            }
        }
        __syncwarp();
    }
    if (lane == 0) {
        red_m[warp] = m;
        red_l[warp] = l;
    }
    red_acc[warp][2 * lane] = acc0;
    red_acc[warp][2 * lane + 1] = acc1;
    __syncthreads();
    if (tid < D) {
        float M = -INFINITY;
        for (int w = 0; w < DEC_WARPS; ++w) M = fmaxf(M, red_m[w]);
        float L2 = 0.0f, o = 0.0f;
        for (int w = 0; w < DEC_WARPS; ++w) {
            const float f = red_m[w] == -INFINITY ? 0.0f : exp2f(red_m[w] - M);
            L2 += red_l[w] * f;
            o += red_acc[w][tid] * f;
        }
        reinterpret_cast<T*>(a.out)[(int64_t)bh * D + tid] = from_f<T>(o / L2);
    }
}

cudaError_t launch_decode(const DecodeArgs& a, bool bf16, cudaStream_t s) {
    if (bf16) {
        const int smem = DEC_WARPS * 2 * 2 * TK * 64 * 2;
        cudaFuncSetAttribute(decode_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        decode_kernel<__nv_bfloat16><<<a.BH, DEC_THREADS, smem, s>>>(a);
    } else {
        const int smem = DEC_WARPS * 2 * 2 * TK * 64 * 4;
        cudaFuncSetAttribute(decode_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        decode_kernel<float><<<a.BH, DEC_THREADS, smem, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace kvm
