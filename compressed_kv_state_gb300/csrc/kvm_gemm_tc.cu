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
// One CTA per 128 x 128 output tile (128 threads, two CTAs per SM): warp 0
// lane 0 issues the TMA loads (128-byte swizzle, 3 stages of 64-wide K
// blocks), warp 1 lane 0 issues the tcgen05 MMAs, then all four warps drain
// tensor memory (thread i = output row i).  Every wait is bounded.
#include <cuda.h>

#include "kvm_internal.cuh"
#include "tc_primitives.cuh"

namespace kvm {
namespace gemm {

using namespace tc;

constexpr int BM = 128, BN = 128, BK = 64, NSTAGE = 3;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int OFF_BAR = NSTAGE * STAGE_BYTES;
constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;  // + alignment slack

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

__global__ void __launch_bounds__(128, 2)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const Args a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    // bars[0, NSTAGE): stage full; [NSTAGE, 2 NSTAGE): stage empty; [2 NSTAGE]: accumulator done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * NSTAGE + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    auto bar = [&](int i) { return smem_u32(bars + i); };

    const int nt = blockIdx.x % a.tiles_n;
    const int mt = blockIdx.x / a.tiles_n;
    const int b = mt / a.tiles_m_per_b;
    const int n0 = (mt % a.tiles_m_per_b) * BM;

    if (tid == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            mbar_init(bar(s), 1);
            mbar_init(bar(NSTAGE + s), 1);
        }
        mbar_init(bar(2 * NSTAGE), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(tmem_slot), BN);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0 && lane == 0) {
        // producer: A and B K-blocks into a ring of NSTAGE stages
        for (int kb = 0; kb < a.kblocks; ++kb) {
            const int s = kb % NSTAGE;
            if (kb >= NSTAGE && !mbar_wait(bar(NSTAGE + s), ((kb / NSTAGE) - 1) & 1, abort_flag, a.status)) break;
            const uint32_t sa = smem_u32(smem + s * STAGE_BYTES), sb = sa + A_BYTES;
            mbar_expect_tx(bar(s), STAGE_BYTES);
            if (a.a_heads)
                tma_load_3d(sa, &tm_a, 0, n0, b * a.H + kb, bar(s));
            else
                tma_load_3d(sa, &tm_a, kb * BK, n0, b, bar(s));
            tma_load_3d(sb, &tm_b, kb * BK, nt * BN, 0, bar(s));
        }
    } else if (warp == 1 && lane == 0) {
        // MMA issuer: D[128 x 128] += A_s[128 x 64] * B_s[128 x 64]^T per stage
        const uint32_t idesc = idesc_bf16(BM, BN, 0, 0);
        bool ok = true;
        for (int kb = 0; kb < a.kblocks && ok; ++kb) {
            const int s = kb % NSTAGE;
            if (!mbar_wait(bar(s), (kb / NSTAGE) & 1, abort_flag, a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(smem + s * STAGE_BYTES), sb = sa + A_BYTES;
#pragma unroll
            for (int ks = 0; ks < BK / 16; ++ks)
                mma_bf16_ss(tmem, sdesc_sw128(sa + ks * 32, 16, 1024), sdesc_sw128(sb + ks * 32, 16, 1024), idesc,
                            (kb | ks) ? 1u : 0u);
            mma_commit(bar(NSTAGE + s));
        }
        mma_commit(bar(2 * NSTAGE));
    }
    __syncwarp();

    // epilogue: thread i drains output row i (TMEM lane i) in 32-column pieces
    const bool done = mbar_wait(bar(2 * NSTAGE), 0, abort_flag, a.status);
    tc_fence_after();
    const int row = tid;
    const int n = n0 + row;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    // tensor-memory loads are warp-wide: the whole warp drains or none of it
    if (__all_sync(0xffffffffu, done && !*abort_flag)) {
        const int Hd = a.H * D;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            const int col0 = nt * BN + c * 32;
            if (col0 >= a.Nout) break;
            uint32_t v[32];
            tmem_ld32(tmem + lane_base + c * 32, v);
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
                for (int i = 0; i < 32; ++i) {
                    const int h = col0 + i - 3 * Hd;
                    if (col0 + i < a.Nout)
                        a.gate[((int64_t)b * a.H + h) * a.N + n] = 1.0f / (1.0f + __expf(-__uint_as_float(v[i])));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        const long long t0 = clock64();
        while (clock64() - t0 < (1ll << 22)) {
        }
    }
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, BN);
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
    const int64_t grid = (int64_t)a.tiles_n * a.tiles_m_per_b * g.B;
    if (grid > 0x7fffffff) return cudaErrorInvalidValue;
    cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    gemm_tc_kernel<<<(unsigned)grid, 128, SMEM_BYTES, s>>>(ma, mb, a);
    return cudaGetLastError();
}

}  // namespace kvm
