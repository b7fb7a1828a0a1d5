// KVM prefill attention on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// "Key-Value Means" (gist.science technical summary), Methodology and Core
// mechanism 4: one softmax over the compressed state's read view (keys zero
// on the rotary dims, read by the unrotated query) and the block-sliding
// window (RoPE on query and keys).  Query p of chunk c sees the state after
// the fold of chunk c - W/C - 1 and the window tokens (c - W/C)*C .. p.
//
// Work unit: a tile of 128 consecutive queries of one (b, h) row (chunks are
// multiples of 128, so a tile never spans two chunks).  The tile's keys come
// in blocks of 128: first ceil(n/128) blocks of the state snapshot, then the
// window from (c - W/C)*C up to the tile's end (the last block is causal).
//
// Persistent CTAs (one per SM, 256 threads) loop over tiles; warp roles:
//   warp 0     TMA producer: Q tile (double-buffered), K/V blocks (3 stages)
//   warp 1     tensor-memory owner and MMA issuer (one thread):
//              S = Q K^T into one of two TMEM S buffers (128 fp32 columns),
//              O += P V into the TMEM O accumulator (64 columns)
//   warps 2-3  RoPE: rotate the Q tile and every window K block in shared
//              memory (128-byte swizzled rows), then hand them to the MMA
//   warps 4-7  softmax: thread i owns query row i (= TMEM lane i); online
//              softmax with lazy rescaling of O (only when the running
//              maximum grows by more than 2^8), P written to shared memory
//              as bf16 in the swizzled K-major layout the MMA reads.
// All mbarrier waits are bounded (about two seconds); on expiry the CTA
// raises the device status word, drains and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kvm_internal.cuh"
#include "tc_primitives.cuh"

namespace kvm {
namespace tc {

constexpr int NS = 3;                 // K/V pipeline stages
constexpr int TILE_BYTES = 128 * 128; // one [128 x 64] bf16 tile
constexpr int OFF_Q = 0;              // 2 Q buffers
constexpr int OFF_K = OFF_Q + 2 * TILE_BYTES;
constexpr int OFF_V = OFF_K + NS * TILE_BYTES;
constexpr int OFF_P = OFF_V + NS * TILE_BYTES;  // 2 P buffers of [128 x 128] bf16
constexpr int OFF_BAR = OFF_P + 2 * 2 * TILE_BYTES;
constexpr int SMEM_BYTES = OFF_BAR + 512 + 1024;  // barriers + alignment slack
constexpr int TMEM_COLS = 512;
constexpr int TM_S0 = 0, TM_O = 256;
constexpr float TAU = 8.0f;  // lazy-rescale threshold (log2 units)

struct TcArgs {
    int64_t N;
    int BH, C, W, M, r;
    int tiles_per_head, ntiles;
    int snap_events;
    const Sched* sched;
    const float2* rope;
    float scale_log2;
    __nv_bfloat16* out;
    int* status;
};

struct Tile {
    int bh, e, n, nst, nwin, nblk;
    int64_t q0, ws;
};

__device__ __forceinline__ Tile tile_of(const TcArgs& a, int id) {
    Tile t;
    t.bh = id / a.tiles_per_head;
    t.q0 = (int64_t)(id % a.tiles_per_head) * 128;
    const int64_t c = t.q0 / a.C, Wc = a.W / a.C;
    t.e = (int)(c - Wc - 1);
    t.n = t.e >= 0 ? a.sched[t.e].n_after : 0;
    t.ws = c - Wc > 0 ? (c - Wc) * a.C : 0;
    t.nst = (t.n + 127) / 128;
    t.nwin = (int)((t.q0 + 128 - t.ws) / 128);
    t.nblk = t.nst + t.nwin;
    return t;
}

// Rotate-half RoPE of one 128-byte swizzled bf16 row in shared memory.
__device__ __forceinline__ void rope_row(uint8_t* row, int row_idx, int64_t pos, const float2* rope,
                                         int half) {
    const float2* cs_row = rope + pos * half;
    const int sw = row_idx & 7;
    for (int x = 0; x < half; ++x) {
        const int xb = x + half;
        __nv_bfloat16* pa = reinterpret_cast<__nv_bfloat16*>(row + ((((x >> 3) ^ sw) << 4) | ((x & 7) << 1)));
        __nv_bfloat16* pb = reinterpret_cast<__nv_bfloat16*>(row + ((((xb >> 3) ^ sw) << 4) | ((xb & 7) << 1)));
        const float2 cs = cs_row[x];
        const float va = __bfloat162float(*pa), vb = __bfloat162float(*pb);
        *pa = __float2bfloat16_rn(va * cs.x - vb * cs.y);
        *pb = __float2bfloat16_rn(vb * cs.x + va * cs.y);
    }
}

__global__ void __launch_bounds__(256, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_sk,
                   const __grid_constant__ CUtensorMap tm_sv, const TcArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    // barrier slots
    enum {
        B_QFULL = 0,              // [2] TMA Q landed
        B_QREADY = 2,             // [2] Q rotated (64 arrivals)
        B_QEMPTY = 4,             // [2] last QK of the tile done
        B_KFULL = 6,              // [NS] TMA K landed
        B_VFULL = B_KFULL + NS,   // [NS] TMA V landed
        B_KREADY = B_VFULL + NS,  // [NS] K rotated (64 arrivals)
        B_KVEMPTY = B_KREADY + NS,// [NS] PV of the stage done
        B_SFULL = B_KVEMPTY + NS, // [2] QK done
        B_PFULL = B_SFULL + 2,    // [2] P written, O rescaled (128 arrivals)
        B_PVDONE = B_PFULL + 2,   // [2] PV done
        B_FINAL = B_PVDONE + 2,   // MMA drain
        NBARS = B_FINAL + 1
    };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    auto bar = [&](int i) { return smem_u32(bars + i); };

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_QFULL + i), 1);
            mbar_init(bar(B_QREADY + i), 64);
            mbar_init(bar(B_QEMPTY + i), 1);
            mbar_init(bar(B_SFULL + i), 1);
            mbar_init(bar(B_PFULL + i), 128);
            mbar_init(bar(B_PVDONE + i), 1);
        }
        for (int s = 0; s < NS; ++s) {
            mbar_init(bar(B_KFULL + s), 1);
            mbar_init(bar(B_VFULL + s), 1);
            mbar_init(bar(B_KREADY + s), 64);
            mbar_init(bar(B_KVEMPTY + s), 1);
        }
        mbar_init(bar(B_FINAL), 1);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sQ = smem_u32(smem + OFF_Q), sK = smem_u32(smem + OFF_K);
    const uint32_t sV = smem_u32(smem + OFF_V), sP = smem_u32(smem + OFF_P);
    const int half = a.r / 2;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int g = 0, tt = 0;
            for (int id = blockIdx.x; id < a.ntiles; id += gridDim.x, ++tt) {
                const Tile T = tile_of(a, id);
                const int qb = tt & 1;
                if (tt >= 2 && !mbar_wait(bar(B_QEMPTY + qb), ((tt >> 1) - 1) & 1, abort_flag, a.status)) break;
                mbar_expect_tx(bar(B_QFULL + qb), TILE_BYTES);
                tma_load_3d(sQ + qb * TILE_BYTES, &tm_q, 0, (int)T.q0, T.bh, bar(B_QFULL + qb));
                bool ok = true;
                for (int j = 0; j < T.nblk; ++j, ++g) {
                    const int s = g % NS;
                    if (g >= NS && !mbar_wait(bar(B_KVEMPTY + s), ((g / NS) - 1) & 1, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(bar(B_KFULL + s), TILE_BYTES);
                    mbar_expect_tx(bar(B_VFULL + s), TILE_BYTES);
                    if (j < T.nst) {
                        const int plane = T.bh * a.snap_events + T.e;
                        tma_load_3d(sK + s * TILE_BYTES, &tm_sk, 0, 128 * j, plane, bar(B_KFULL + s));
                        tma_load_3d(sV + s * TILE_BYTES, &tm_sv, 0, 128 * j, plane, bar(B_VFULL + s));
                    } else {
                        const int key0 = (int)(T.ws + 128 * (j - T.nst));
                        tma_load_3d(sK + s * TILE_BYTES, &tm_k, 0, key0, T.bh, bar(B_KFULL + s));
                        tma_load_3d(sV + s * TILE_BYTES, &tm_v, 0, key0, T.bh, bar(B_VFULL + s));
                    }
                }
                if (!ok) break;
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc_qk = idesc_bf16(128, 128, 0, 0);
            const uint32_t idesc_pv = idesc_bf16(128, 64, 0, 1);
            int g = 0, tt = 0;
            bool ok = true;
            for (int id = blockIdx.x; id < a.ntiles && ok; id += gridDim.x, ++tt) {
                const Tile T = tile_of(a, id);
                const int qb = tt & 1;
                if (!mbar_wait(bar(B_QREADY + qb), (tt >> 1) & 1, abort_flag, a.status)) break;
                tc_fence_after();
                const int ks_state = min(a.r / 16, 3);
                auto issue_qk = [&](int j, int gq) -> bool {
                    const int s = gq % NS, sb = gq & 1;
                    if (!mbar_wait(bar(B_KREADY + s), (gq / NS) & 1, abort_flag, a.status)) return false;
                    tc_fence_after();
                    const int ks0 = j < T.nst ? ks_state : 0;
                    for (int ks = ks0; ks < 4; ++ks) {
                        const uint64_t ad = sdesc_sw128(sQ + qb * TILE_BYTES + ks * 32, 16, 1024);
                        const uint64_t bd = sdesc_sw128(sK + s * TILE_BYTES + ks * 32, 16, 1024);
                        mma_bf16_ss(tmem + TM_S0 + sb * 128, ad, bd, idesc_qk, ks > ks0);
                    }
                    mma_commit(bar(B_SFULL + sb));
                    return true;
                };
                if (!issue_qk(0, g)) { ok = false; break; }
                for (int j = 0; j < T.nblk; ++j) {
                    const int gj = g + j;
                    if (j + 1 < T.nblk) {
                        if (!issue_qk(j + 1, gj + 1)) { ok = false; break; }
                    } else {
                        mma_commit(bar(B_QEMPTY + qb));
                    }
                    const int s = gj % NS, pb = gj & 1;
                    if (!mbar_wait(bar(B_PFULL + pb), (gj >> 1) & 1, abort_flag, a.status) ||
                        !mbar_wait(bar(B_VFULL + s), (gj / NS) & 1, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    for (int ks = 0; ks < 8; ++ks) {
                        const uint64_t ad = sdesc_sw128(sP + pb * 2 * TILE_BYTES + (ks >> 2) * TILE_BYTES + (ks & 3) * 32, 16, 1024);
                        const uint64_t bd = sdesc_sw128(sV + s * TILE_BYTES + ks * 2048, TILE_BYTES, 1024);
                        mma_bf16_ss(tmem + TM_O, ad, bd, idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
                    }
                    mma_commit(bar(B_PVDONE + pb));
                    mma_commit(bar(B_KVEMPTY + s));
                }
                g += T.nblk;
            }
            // drain: every MMA issued above has completed once this arrives
            mma_commit(bar(B_FINAL));
            mbar_wait(bar(B_FINAL), 0, abort_flag, nullptr);
        }
    } else if (warp < 4) {
        // --------------------------------------------------------------- RoPE
        const int rt = tid - 64;
        int g = 0, tt = 0;
        for (int id = blockIdx.x; id < a.ntiles; id += gridDim.x, ++tt) {
            const Tile T = tile_of(a, id);
            const int qb = tt & 1;
            if (!mbar_wait(bar(B_QFULL + qb), (tt >> 1) & 1, abort_flag, a.status)) break;
            if (half > 0) {
                for (int row = rt; row < 128; row += 64) {
                    const int64_t pos = T.q0 + row;
                    if (pos < a.N) rope_row(smem + OFF_Q + qb * TILE_BYTES + row * 128, row, pos, a.rope, half);
                }
            }
            fence_proxy_async();
            mbar_arrive(bar(B_QREADY + qb));
            bool ok = true;
            for (int j = 0; j < T.nblk; ++j, ++g) {
                const int s = g % NS;
                if (!mbar_wait(bar(B_KFULL + s), (g / NS) & 1, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                if (j >= T.nst && half > 0) {
                    const int64_t key0 = T.ws + 128 * (j - T.nst);
                    for (int row = rt; row < 128; row += 64) {
                        const int64_t pos = key0 + row;
                        if (pos < a.N) rope_row(smem + OFF_K + s * TILE_BYTES + row * 128, row, pos, a.rope, half);
                    }
                }
                fence_proxy_async();
                mbar_arrive(bar(B_KREADY + s));
            }
            if (!ok) break;
        }
    } else {
        // ------------------------------------------------------------ softmax
        const int row = tid - 128;                 // query row = TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        int g = 0;
        bool ok = true;
        for (int id = blockIdx.x; id < a.ntiles && ok; id += gridDim.x) {
            const Tile T = tile_of(a, id);
            const int64_t p = T.q0 + row;
            float m_used = -INFINITY, l = 0.0f;
            for (int j = 0; j < T.nblk; ++j) {
                const int gj = g + j, sb = gj & 1;
                if (!mbar_wait(bar(B_SFULL + sb), (gj >> 1) & 1, abort_flag, a.status)) { ok = false; break; }
                tc_fence_after();
                uint32_t sr[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_base + TM_S0 + sb * 128 + c * 32, sr[c]);
                tmem_wait_ld();
                const bool is_state = j < T.nst;
                const int64_t key0 = is_state ? 0 : T.ws + 128 * (j - T.nst);
                // limit: columns < lim are valid
                int lim;
                if (is_state) lim = min(128, T.n - 128 * j);
                else lim = (p - key0 + 1) < 128 ? (int)(p - key0 + 1) : 128;
                float mblk = -INFINITY;
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int x = 0; x < 32; ++x) {
                        const int col = c * 32 + x;
                        float v = __uint_as_float(sr[c][x]) * a.scale_log2;
                        v = col < lim ? v : -INFINITY;
                        sr[c][x] = __float_as_uint(v);
                        mblk = fmaxf(mblk, v);
                    }
                bool rescale = false;
                float alpha = 1.0f;
                if (mblk > m_used) {
                    if (m_used == -INFINITY) {
                        m_used = mblk;
                    } else if (mblk > m_used + TAU) {
                        alpha = ex2(m_used - mblk);
                        m_used = mblk;
                        rescale = true;
                    }
                }
                l *= alpha;
                uint32_t pk[64];
                float rs = 0.0f;
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int x = 0; x < 32; x += 2) {
                        const float p0 = ex2(__uint_as_float(sr[c][x]) - m_used);
                        const float p1 = ex2(__uint_as_float(sr[c][x + 1]) - m_used);
                        rs += p0 + p1;
                        __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
                        pk[(c * 32 + x) >> 1] = *reinterpret_cast<uint32_t*>(&h);
                    }
                l += rs;
                if (rescale) {
                    // O holds blocks < j: wait for the last PV, then scale it in place
                    if (!mbar_wait(bar(B_PVDONE + ((gj - 1) & 1)), ((gj - 1) >> 1) & 1, abort_flag, a.status)) { ok = false; break; }
                    tc_fence_after();
                    uint32_t o[2][32];
                    tmem_ld32(tmem + lane_base + TM_O, o[0]);
                    tmem_ld32(tmem + lane_base + TM_O + 32, o[1]);
                    tmem_wait_ld();
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int x = 0; x < 32; ++x) o[h][x] = __float_as_uint(__uint_as_float(o[h][x]) * alpha);
                    tmem_st32(tmem + lane_base + TM_O, o[0]);
                    tmem_st32(tmem + lane_base + TM_O + 32, o[1]);
                    tmem_wait_st();
                }
                // the P buffer was last read by the PV of block gj - 2
                if (gj >= 2 && !mbar_wait(bar(B_PVDONE + sb), ((gj - 2) >> 1) & 1, abort_flag, a.status)) { ok = false; break; }
                uint8_t* prow = smem + OFF_P + sb * 2 * TILE_BYTES + row * 128;
#pragma unroll
                for (int ch = 0; ch < 16; ++ch) {
                    const int hsub = ch >> 3, c8 = ch & 7;
                    uint4 val = make_uint4(pk[ch * 4 + 0], pk[ch * 4 + 1], pk[ch * 4 + 2], pk[ch * 4 + 3]);
                    *reinterpret_cast<uint4*>(prow + hsub * TILE_BYTES + ((c8 ^ (row & 7)) << 4)) = val;
                }
                fence_proxy_async();
                tc_fence_before();
                mbar_arrive(bar(B_PFULL + sb));
            }
            if (!ok) break;
            // epilogue: O / l for this tile
            const int gl = g + T.nblk - 1;
            if (!mbar_wait(bar(B_PVDONE + (gl & 1)), (gl >> 1) & 1, abort_flag, a.status)) { ok = false; break; }
            tc_fence_after();
            uint32_t o[2][32];
            tmem_ld32(tmem + lane_base + TM_O, o[0]);
            tmem_ld32(tmem + lane_base + TM_O + 32, o[1]);
            tmem_wait_ld();
            tc_fence_before();
            if (p < a.N) {
                const float il = 1.0f / l;
                uint4* dst = reinterpret_cast<uint4*>(a.out + ((int64_t)T.bh * a.N + p) * D);
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int x = 0; x < 32; x += 8) {
                        uint32_t w[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(o[h][x + 2 * u]) * il,
                                                                      __uint_as_float(o[h][x + 2 * u + 1]) * il);
                            w[u] = *reinterpret_cast<uint32_t*>(&b2);
                        }
                        dst[(h * 32 + x) >> 3] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
            }
            g += T.nblk;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        // let copies still in flight land before the shared memory is released
        const long long t0 = clock64();
        while (clock64() - t0 < (1ll << 22)) {
        }
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host

static PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace tc

// 3-D bf16 map over [planes][rows][64] with a 128 x 64 box, 128-byte swizzle.
bool make_tmap_bf16_3d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t planes) {
    using namespace tc;
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {64, rows, planes};
    cuuint64_t strides[2] = {64 * 2, rows * 64 * 2};
    cuuint32_t box[3] = {64, 128, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool attn_tc_supported(const AttnArgs& a, bool bf16) {
    return bf16 && a.C % 128 == 0 && a.N > 0;
}

cudaError_t launch_attn_tc(const AttnArgs& a, int* status, cudaStream_t s) {
    using namespace tc;
    CUtensorMap mq, mk, mv, msk, msv;
    const uint64_t BH = (uint64_t)a.BH;
    const uint64_t planes_snap = BH * (uint64_t)(a.snap_events > 0 ? a.snap_events : 1);
    if (!make_tmap_bf16_3d(&mq, a.q, (uint64_t)a.N, BH) || !make_tmap_bf16_3d(&mk, a.k, (uint64_t)a.N, BH) ||
        !make_tmap_bf16_3d(&mv, a.v, (uint64_t)a.N, BH) ||
        !make_tmap_bf16_3d(&msk, a.snap_k, (uint64_t)a.M, planes_snap) ||
        !make_tmap_bf16_3d(&msv, a.snap_v, (uint64_t)a.M, planes_snap))
        return cudaErrorInvalidValue;
    TcArgs t;
    t.N = a.N;
    t.BH = a.BH;
    t.C = a.C;
    t.W = a.W;
    t.M = a.M;
    t.r = a.r;
    t.tiles_per_head = (int)((a.N + 127) / 128);
    t.ntiles = t.tiles_per_head * a.BH;
    t.snap_events = a.snap_events;
    t.sched = a.sched;
    t.rope = a.rope;
    t.scale_log2 = a.scale_log2;
    t.out = reinterpret_cast<__nv_bfloat16*>(a.out);
    t.status = status;
    static int nsm = 0;
    if (nsm == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    }
    const int grid = t.ntiles < nsm ? t.ntiles : nsm;
    cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    attn_tc_kernel<<<grid, 256, SMEM_BYTES, s>>>(mq, mk, mv, msk, msv, t);
    return cudaGetLastError();
}

}  // namespace kvm
