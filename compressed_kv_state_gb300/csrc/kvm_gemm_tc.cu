// Projections of the whole KVM attention layer on the tensor cores.
//
// "Key-Value Means" (gist.science technical summary), Methodology: the layer
// projects its input to queries, keys, values and a data-dependent merge gate,
// runs the KVM attention per head, and projects the heads back.  Both
// projections are C = A * B^T with A [rows, K] and B [Nout, K] (the linear
// layer's weight layout), both K-major bf16, accumulated in fp32 in tensor
// memory, with the epilogue fused:
//   - input projection: columns [0, 3*H*64) are q, k, v of head h, written
//     bf16 straight into [B, H, N, 64]; columns [3*H*64, 3*H*64 + H) are the
//     merge-gate logits of head h, written as sigmoid(logit) fp32 [B, H, N];
//   - output projection: A is the attention output [B, H, N, 64] read
//     head by head (K-block h = head h), C is written bf16 [B, N, Nout].
// Persistent: one CTA per SM walks its share of the 128 x 256 output tiles.
// Warp 0 lane 0 issues the TMA loads (128-byte swizzle, a ring of 4 stages of
// 64-wide K blocks, running across tile boundaries), warp 1 lane 0 issues the
// tcgen05 MMAs (M 128, N 256) into one of two TMEM accumulators (tile i uses
// accumulator i % 2; together they fill the 512 columns), and warps 2-5 drain
// the other accumulator meanwhile (thread = output row = TMEM lane), so a
// tile's epilogue overlaps the next tile's MMAs.  Every wait is bounded.
#include <cuda.h>

#include "kvm_internal.cuh"
#include "tc_primitives.cuh"

namespace kvm {
namespace gemm {

using namespace tc;

constexpr int BM = 128, BN = 256, BK = 64, NSTAGE = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int OFF_BAR = NSTAGE * STAGE_BYTES;
constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;  // + alignment slack
constexpr int EPI_THREADS = 128;                  // warps 2-5
constexpr int THREADS = 64 + EPI_THREADS;

struct Args {
    int B, N, H;
    int K, Nout, kblocks;
    int tiles_m_per_b, tiles_n;
    int a_heads;  // A from [B*H, N, 64] planes: K-block kb is head kb
    int epi;      // 0: q/k/v/gate scatter, 1: row-major output
    __nv_bfloat16* q;
    __nv_bfloat16* k;
    __nv_bfloat16* v;
    float* gate;
    __nv_bfloat16* y;
    int* status;
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// 32 consecutive fp32 columns -> 32 bf16 (64 contiguous bytes)
__device__ __forceinline__ void store32_bf16(__nv_bfloat16* dst, const uint32_t (&v)[32]) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int c = 0; c < 4; ++c)
        d4[c] = make_uint4(pack_bf16(__uint_as_float(v[8 * c]), __uint_as_float(v[8 * c + 1])),
                           pack_bf16(__uint_as_float(v[8 * c + 2]), __uint_as_float(v[8 * c + 3])),
                           pack_bf16(__uint_as_float(v[8 * c + 4]), __uint_as_float(v[8 * c + 5])),
                           pack_bf16(__uint_as_float(v[8 * c + 6]), __uint_as_float(v[8 * c + 7])));
}

__global__ void __launch_bounds__(THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const Args a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    // bars: [0, NSTAGE) stage full, [NSTAGE, 2 NSTAGE) stage empty,
    // [2 NSTAGE, +2) accumulator full, [2 NSTAGE + 2, +2) accumulator drained
    constexpr int B_FULL = 0, B_EMPTY = NSTAGE, B_ACCF = 2 * NSTAGE, B_ACCE = 2 * NSTAGE + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * NSTAGE + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    auto bar = [&](int i) { return smem_u32(bars + i); };
    const int ntiles = a.tiles_n * a.tiles_m_per_b * a.B;

    if (tid == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(bar(B_FULL + s), 1);
            mbar_init(bar(B_EMPTY + s), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_ACCF + i), 1);
            mbar_init(bar(B_ACCE + i), EPI_THREADS);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(tmem_slot), 2 * BN);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // producer: A and B K-blocks of every tile of this CTA through a ring of NSTAGE stages
            int g = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
                const int nt = t % a.tiles_n, mt = t / a.tiles_n;
                const int b = mt / a.tiles_m_per_b, n0 = (mt % a.tiles_m_per_b) * BM;
                for (int kb = 0; kb < a.kblocks; ++kb, ++g) {
                    const int s = g % NSTAGE;
                    if (g >= NSTAGE && !mbar_wait(bar(B_EMPTY + s), ((g / NSTAGE) - 1) & 1, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = smem_u32(smem + s * STAGE_BYTES), sb = sa + A_BYTES;
                    mbar_expect_tx(bar(B_FULL + s), STAGE_BYTES);
                    if (a.a_heads)
                        tma_load_3d(sa, &tm_a, 0, n0, b * a.H + kb, bar(B_FULL + s));
                    else
                        tma_load_3d(sa, &tm_a, kb * BK, n0, b, bar(B_FULL + s));
                    tma_load_3d(sb, &tm_b, kb * BK, nt * BN, 0, bar(B_FULL + s));
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // MMA issuer: tile i accumulates into TMEM columns (i & 1) * BN once the
            // epilogue has drained what tile i - 2 left there
            const uint32_t idesc = idesc_bf16(BM, BN, 0, 0);
            int g = 0, i = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++i) {
                const int acc = i & 1;
                if (i >= 2 && !mbar_wait(bar(B_ACCE + acc), ((i >> 1) - 1) & 1, abort_flag, a.status)) break;
                tc_fence_after();
                for (int kb = 0; kb < a.kblocks; ++kb, ++g) {
                    const int s = g % NSTAGE;
                    if (!mbar_wait(bar(B_FULL + s), (g / NSTAGE) & 1, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + s * STAGE_BYTES), sb = sa + A_BYTES;
#pragma unroll
                    for (int ks = 0; ks < BK / 16; ++ks)
                        mma_bf16_ss(tmem + acc * BN, sdesc_sw128(sa + ks * 32, 16, 1024),
                                    sdesc_sw128(sb + ks * 32, 16, 1024), idesc, (kb | ks) ? 1u : 0u);
                    mma_commit(bar(B_EMPTY + s));
                }
                mma_commit(bar(B_ACCF + acc));
            }
        }
    } else {
        // epilogue warps 2-5: warp w drains TMEM lanes 32 * (w % 4) .. + 31 (output rows)
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const int Hd = a.H * D;
        int i = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
            const int acc = i & 1;
            const bool ok = mbar_wait(bar(B_ACCF + acc), (i >> 1) & 1, abort_flag, a.status);
            // tensor-memory loads are warp-wide: the whole warp drains or none of it
            if (!__all_sync(0xffffffffu, ok && !*abort_flag)) break;
            tc_fence_after();
            const int nt = t % a.tiles_n, mt = t / a.tiles_n;
            const int b = mt / a.tiles_m_per_b, n = (mt % a.tiles_m_per_b) * BM + row;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                const int col0 = nt * BN + c * 32;
                if (col0 >= a.Nout) break;
                uint32_t v[32];
                tmem_ld32(tmem + lane_base + acc * BN + c * 32, v);
                tmem_wait_ld();
                if (n >= a.N) continue;
                if (a.epi == 1) {
                    store32_bf16(a.y + ((int64_t)b * a.N + n) * a.Nout + col0, v);
                } else if (col0 < 3 * Hd) {
                    const int which = col0 / Hd, h = (col0 % Hd) / D, x0 = col0 % D;
                    __nv_bfloat16* dst = which == 0 ? a.q : (which == 1 ? a.k : a.v);
                    store32_bf16(dst + (((int64_t)b * a.H + h) * a.N + n) * D + x0, v);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int h = col0 + j - 3 * Hd;
                        if (col0 + j < a.Nout)
                            a.gate[((int64_t)b * a.H + h) * a.N + n] = 1.0f / (1.0f + __expf(-__uint_as_float(v[j])));
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(bar(B_ACCE + acc));
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        // let copies and MMAs still in flight finish before shared and tensor memory go
        const long long t0 = clock64();
        while (clock64() - t0 < (1ll << 22)) {
        }
    }
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 2 * BN);
    }
}

}  // namespace gemm

bool make_tmap_bf16_rows(CUtensorMap* m, const void* base, uint64_t row_elems, uint64_t rows, uint64_t planes,
                         uint32_t box_rows);

cudaError_t launch_gemm_tc(const GemmSpec& g, cudaStream_t s) {
    using namespace gemm;
    if (g.K % BK != 0 || g.Nout <= 0 || g.N <= 0) return cudaErrorInvalidValue;
    CUtensorMap ma, mb;
    const bool ok_a = g.a_heads ? make_tmap_bf16_rows(&ma, g.a, 64, (uint64_t)g.N, (uint64_t)g.B * g.H, BM)
                                : make_tmap_bf16_rows(&ma, g.a, (uint64_t)g.K, (uint64_t)g.N, (uint64_t)g.B, BM);
    if (!ok_a || !make_tmap_bf16_rows(&mb, g.w, (uint64_t)g.K, (uint64_t)g.Nout, 1, BN)) return cudaErrorInvalidValue;
    Args a{};
    a.B = g.B;
    a.N = (int)g.N;
    a.H = g.H;
    a.K = g.K;
    a.Nout = g.Nout;
    a.kblocks = g.K / BK;
    a.tiles_m_per_b = (int)((g.N + BM - 1) / BM);
    a.tiles_n = (g.Nout + BN - 1) / BN;
    a.a_heads = g.a_heads;
    a.epi = g.epi;
    a.q = static_cast<__nv_bfloat16*>(g.q);
    a.k = static_cast<__nv_bfloat16*>(g.k);
    a.v = static_cast<__nv_bfloat16*>(g.v);
    a.gate = g.gate;
    a.y = static_cast<__nv_bfloat16*>(g.y);
    a.status = g.status;
    const int64_t tiles = (int64_t)a.tiles_n * a.tiles_m_per_b * g.B;
    if (tiles > 0x7fffffff) return cudaErrorInvalidValue;
    int dev = 0, nsm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    const int grid = (int)(tiles < nsm ? tiles : (nsm > 0 ? nsm : 1));
    cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    gemm_tc_kernel<<<grid, THREADS, SMEM_BYTES, s>>>(ma, mb, a);
    return cudaGetLastError();
}

}  // namespace kvm
