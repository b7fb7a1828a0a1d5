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
// in blocks of 64: first ceil(n/64) blocks of the state snapshot, then the
// window from (c - W/C)*C up to the tile's end (the last block is causal).
//
// Persistent CTAs (two per SM, 256 threads, 97 KB shared memory and 256 TMEM
// columns each, so the tensor core alternates between two tiles) take tiles in
// turns, either statically strided or claimed from a counter shared by several
// launches; warp roles:
//   warp 0     TMA producer: claims the tile, loads Q and the K/V blocks
//              (3 stages)
//   warp 1     tensor-memory owner and MMA issuer (one thread):
//              S = Q K^T into one of two 64-column TMEM S buffers, issued for
//              block j+1 before O += P V of block j (O: 64 columns)
//   warps 2-3  RoPE: rotate the Q tile in shared memory (128-byte swizzled
//              rows) and hand it to the MMA; window keys normally arrive
//              already rotated (k_rot, rotated once per key by
//              rope_keys_kernel), and only without that copy do these warps
//              rotate each window K block as well
//   warps 4-7  softmax: thread i owns query row i (= TMEM lane i); one pass
//              over the 64-column S row, lazy rescaling of O (only when the
//              running maximum grows by more than 2^8), P written to shared
//              memory as bf16 in the swizzled K-major layout the MMA reads.
// All mbarrier waits are bounded (about two seconds); on expiry the CTA
// raises the device status word, drains and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>

#include "kvm_internal.cuh"
#include "tc_primitives.cuh"

namespace kvm {
namespace tc {

constexpr int NS = 3;                 // K/V pipeline stages
constexpr int KB = 64;                // keys per block
constexpr int Q_BYTES = 128 * 128;    // Q tile [128 x 64] bf16
constexpr int KV_BYTES = KB * 128;    // K or V block [64 x 64] bf16
constexpr int P_BYTES = 128 * 128;    // P block [128 x 64] bf16
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + Q_BYTES;
constexpr int OFF_V = OFF_K + NS * KV_BYTES;
constexpr int OFF_P = OFF_V + NS * KV_BYTES;    // 2 P buffers
constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;
constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;  // 97.25 KB with alignment slack: two CTAs per SM
constexpr int TMEM_COLS = 256;
constexpr int TM_S = 0, TM_O = 128;             // S buffers at columns 0 and 64
constexpr float TAU = 8.0f;  // lazy-rescale threshold (log2 units)

#ifdef KVM_PROBE
static __device__ unsigned long long g_probe_attn[64];
#endif

struct TcArgs {
    int64_t N;
    int BH, C, W, M, r;
    int tiles_per_head, ntiles;
    int k_rotated;   // window keys arrive rotated (no RoPE on K in the kernel)
    int* tile_ctr;   // dynamic claiming: one counter per range (nullptr: static striding)
    int n_ranges;
    int range_end[AttnArgs::MAX_RANGES];
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

// Tiles are numbered query-tile-major: number id is query tile id / BH of row
// id % BH, so every prefix of the numbering is a set of whole chunks of all rows
// (the order in which the fold chain makes their state snapshots available).
__device__ __forceinline__ Tile tile_of(const TcArgs& a, int id) {
    Tile t;
    t.bh = id % a.BH;
    t.q0 = (int64_t)(id / a.BH) * 128;
    const int64_t c = t.q0 / a.C, Wc = a.W / a.C;
    t.e = (int)(c - Wc - 1);
    t.n = t.e >= 0 ? a.sched[t.e].n_after : 0;
    t.ws = c - Wc > 0 ? (c - Wc) * a.C : 0;
    t.nst = (t.n + KB - 1) / KB;
    t.nwin = (int)((t.q0 + 128 - t.ws) / KB);
    t.nblk = t.nst + t.nwin;
    return t;
}

// The tile a CTA processes in its tt-th turn, or -1 when it is done.  Dynamic
// claiming: the next tile of the first range (from the CTA's cursor *range on)
// that is not exhausted, one atomicAdd per claim (a compare-and-swap loop on a
// shared counter collapses under contention from hundreds of CTAs).  Static:
// blockIdx.x + tt * gridDim.x.
__device__ __forceinline__ int next_tile(const TcArgs& a, int tt, int* range) {
    if (a.tile_ctr) {
        for (; *range < a.n_ranges; ++*range) {
            const int r = *range;
            const int lo = r > 0 ? a.range_end[r - 1] : 0;
            const int id = lo + atomicAdd(a.tile_ctr + r, 1);
            if (id < a.range_end[r]) return id;
        }
        return -1;
    }
    const int64_t id = blockIdx.x + (int64_t)tt * gridDim.x;
    return id < a.ntiles ? (int)id : -1;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
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

// Same rotation when half is a multiple of 8: dims [0, half) and [half, 2*half)
// are whole 16-byte chunks, so a row is rotated with vector shared-memory
// accesses and vector loads of the (cos, sin) table.
__device__ __forceinline__ void rope_row_vec(uint8_t* row, int row_idx, int64_t pos, const float2* rope,
                                             int half) {
    const float4* tab = reinterpret_cast<const float4*>(rope + pos * half);
    const int sw = row_idx & 7;
    const int hc = half >> 3;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        if (c >= hc) break;
        uint4* pa = reinterpret_cast<uint4*>(row + ((c ^ sw) << 4));
        uint4* pb = reinterpret_cast<uint4*>(row + (((c + hc) ^ sw) << 4));
        // element e of the chunk is pair 8c + e: float4 4c + e/2 holds pairs 8c + 2(e/2) (x = cos,
        // y = sin) and 8c + 2(e/2) + 1 (z = cos, w = sin)
        const float4 t0 = tab[4 * c], t1 = tab[4 * c + 1], t2 = tab[4 * c + 2], t3 = tab[4 * c + 3];
        const float ce[8] = {t0.x, t0.z, t1.x, t1.z, t2.x, t2.z, t3.x, t3.z};
        const float se[8] = {t0.y, t0.w, t1.y, t1.w, t2.y, t2.w, t3.y, t3.w};
        uint4 A = *pa, B = *pb;
        __nv_bfloat162* a2 = reinterpret_cast<__nv_bfloat162*>(&A);
        __nv_bfloat162* b2 = reinterpret_cast<__nv_bfloat162*>(&B);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float2 av = __bfloat1622float2(a2[u]), bv = __bfloat1622float2(b2[u]);
            const float c0 = ce[2 * u], c1 = ce[2 * u + 1], s0 = se[2 * u], s1 = se[2 * u + 1];
            a2[u] = __floats2bfloat162_rn(av.x * c0 - bv.x * s0, av.y * c1 - bv.y * s1);
            b2[u] = __floats2bfloat162_rn(bv.x * c0 + av.x * s0, bv.y * c1 + av.y * s1);
        }
        *pa = A;
        *pb = B;
    }
}

__global__ void __launch_bounds__(256, 2)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_sk,
                   const __grid_constant__ CUtensorMap tm_sv, const TcArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned tiles for the 128-byte swizzle (the slack is part of the request)
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    enum {
        B_QFULL = 0,               // TMA Q landed
        B_QREADY = 1,              // Q rotated (64 arrivals)
        B_QEMPTY = 2,              // last QK of the tile done
        B_KFULL = 3,               // [NS] TMA K landed
        B_VFULL = B_KFULL + NS,    // [NS] TMA V landed
        B_KREADY = B_VFULL + NS,   // [NS] K rotated (64 arrivals)
        B_KVEMPTY = B_KREADY + NS, // [NS] PV of the stage done
        B_SFULL = B_KVEMPTY + NS,  // [2] QK done
        B_PFULL = B_SFULL + 2,     // [2] S consumed, P written, O rescaled (128 arrivals)
        B_PVDONE = B_PFULL + 2,    // [2] PV done
        B_FINAL = B_PVDONE + 2,    // MMA drain
        B_TILE = B_FINAL + 1,      // [4] tile number of turn tt published (ring of 4)
        NBARS = B_TILE + 4
    };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* tile_ring = reinterpret_cast<volatile int*>(tmem_slot + 2);
    auto bar = [&](int i) { return smem_u32(bars + i); };
    // The producer publishes the tile of turn tt in ring slot tt % 4; the other roles
    // read it after the slot's barrier.  A slot is rewritten four turns later, when
    // every role has moved past that turn: the producer claims turn tt only after the
    // last QK MMA of turn tt - 1, which follows the rotation of its Q (RoPE warps in
    // turn tt - 1) and the softmax of a block of turn tt - 2 or later.
    auto tile_wait = [&](int tt) -> int {
        if (!mbar_wait(bar(B_TILE + (tt & 3)), (tt >> 2) & 1, abort_flag, a.status)) return -1;
        return tile_ring[tt & 3];
    };

    if (tid == 0) {
        mbar_init(bar(B_QFULL), 1);
        mbar_init(bar(B_QREADY), 64);
        mbar_init(bar(B_QEMPTY), 1);
        for (int i = 0; i < 2; ++i) {
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
        for (int i = 0; i < 4; ++i) mbar_init(bar(B_TILE + i), 1);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
#ifdef KVM_PROBE
    unsigned probe_sm = 0;
    if (tid == 0) {
        if (blockIdx.x == 0) g_probe_attn[31] = gridDim.x;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(probe_sm));
        const unsigned long long now = atomicAdd(&g_probe_attn[32 + (probe_sm & 31)], 1ull) + 1;
        atomicMax(&g_probe_attn[29], now);
    }
#endif
    const uint32_t tmem = *tmem_slot;
    const uint32_t sQ = smem_u32(smem + OFF_Q), sK = smem_u32(smem + OFF_K);
    const uint32_t sV = smem_u32(smem + OFF_V), sP = smem_u32(smem + OFF_P);
    const int half = a.r / 2;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            KVM_PROBE_DECL(3)
            KVM_PROBE_START()
            int g = 0, range = 0;
            for (int tt = 0;; ++tt) {
                KVM_PROBE_LAP(2)
                if (tt >= 1 && !mbar_wait(bar(B_QEMPTY), (tt - 1) & 1, abort_flag, a.status)) break;
                KVM_PROBE_LAP(0)
                const int id = next_tile(a, tt, &range);
                tile_ring[tt & 3] = id;
                mbar_arrive(bar(B_TILE + (tt & 3)));
                if (id < 0) break;
                const Tile T = tile_of(a, id);
                mbar_expect_tx(bar(B_QFULL), Q_BYTES);
                tma_load_3d(sQ, &tm_q, 0, (int)T.q0, T.bh, bar(B_QFULL));
                bool ok = true;
                for (int j = 0; j < T.nblk; ++j, ++g) {
                    const int s = g % NS;
                    KVM_PROBE_LAP(2)
                    if (g >= NS && !mbar_wait(bar(B_KVEMPTY + s), ((g / NS) - 1) & 1, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    KVM_PROBE_LAP(1)
                    mbar_expect_tx(bar(B_KFULL + s), KV_BYTES);
                    mbar_expect_tx(bar(B_VFULL + s), KV_BYTES);
                    if (j < T.nst) {
                        const int plane = T.bh * a.snap_events + T.e;
                        tma_load_3d(sK + s * KV_BYTES, &tm_sk, 0, KB * j, plane, bar(B_KFULL + s));
                        tma_load_3d(sV + s * KV_BYTES, &tm_sv, 0, KB * j, plane, bar(B_VFULL + s));
                    } else {
                        const int key0 = (int)(T.ws + KB * (j - T.nst));
                        tma_load_3d(sK + s * KV_BYTES, &tm_k, 0, key0, T.bh, bar(B_KFULL + s));
                        tma_load_3d(sV + s * KV_BYTES, &tm_v, 0, key0, T.bh, bar(B_VFULL + s));
                    }
                }
                if (!ok) break;
            }
            KVM_PROBE_LAP(2)
            KVM_PROBE_FLUSH(g_probe_attn, 0, 3)
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc_qk = idesc_bf16(128, KB, 0, 0);
            const uint32_t idesc_pv = idesc_bf16(128, 64, 0, 1);
            const int ks_state = min(a.r / 16, 3);
            KVM_PROBE_DECL(5)
            KVM_PROBE_START()
            int g = 0;
            bool ok = true;
            for (int tt = 0; ok; ++tt) {
                const int id = tile_wait(tt);
                if (id < 0) break;
                const Tile T = tile_of(a, id);
                KVM_PROBE_LAP(4)
                if (!mbar_wait(bar(B_QREADY), tt & 1, abort_flag, a.status)) break;
                KVM_PROBE_LAP(0)
                tc_fence_after();
                auto issue_qk = [&](int j, int gq) -> bool {
                    const int s = gq % NS, sb = gq & 1;
                    KVM_PROBE_LAP(4)
                    if (!mbar_wait(bar(B_KREADY + s), (gq / NS) & 1, abort_flag, a.status)) return false;
                    KVM_PROBE_LAP(1)
                    tc_fence_after();
                    const int ks0 = j < T.nst ? ks_state : 0;
                    for (int ks = ks0; ks < 4; ++ks) {
                        const uint64_t ad = sdesc_sw128(sQ + ks * 32, 16, 1024);
                        const uint64_t bd = sdesc_sw128(sK + s * KV_BYTES + ks * 32, 16, 1024);
                        mma_bf16_ss(tmem + TM_S + sb * KB, ad, bd, idesc_qk, ks > ks0);
                    }
                    mma_commit(bar(B_SFULL + sb));
                    return true;
                };
                if (!issue_qk(0, g)) { ok = false; break; }
                for (int j = 0; j < T.nblk; ++j) {
                    const int gj = g + j, s = gj % NS, pb = gj & 1;
                    // S buffer of block gj + 1 last held block gj - 1, consumed before its P was published
                    if (j + 1 < T.nblk) {
                        if (!issue_qk(j + 1, gj + 1)) { ok = false; break; }
                    } else {
                        mma_commit(bar(B_QEMPTY));
                    }
                    KVM_PROBE_LAP(4)
                    if (!mbar_wait(bar(B_PFULL + pb), (gj >> 1) & 1, abort_flag, a.status)) { ok = false; break; }
                    KVM_PROBE_LAP(2)
                    if (!mbar_wait(bar(B_VFULL + s), (gj / NS) & 1, abort_flag, a.status)) { ok = false; break; }
                    KVM_PROBE_LAP(3)
                    tc_fence_after();
                    for (int ks = 0; ks < KB / 16; ++ks) {
                        const uint64_t ad = sdesc_sw128(sP + pb * P_BYTES + ks * 32, 16, 1024);
                        const uint64_t bd = sdesc_sw128(sV + s * KV_BYTES + ks * 2048, KV_BYTES, 1024);
                        mma_bf16_ss(tmem + TM_O, ad, bd, idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
                    }
                    mma_commit(bar(B_PVDONE + pb));
                    mma_commit(bar(B_KVEMPTY + s));
                }
                g += T.nblk;
            }
            KVM_PROBE_LAP(4)
            KVM_PROBE_FLUSH(g_probe_attn, 3, 5)
            mma_commit(bar(B_FINAL));
            mbar_wait(bar(B_FINAL), 0, abort_flag, nullptr);
        }
    } else if (warp < 4) {
        // --------------------------------------------------------------- RoPE
        const int rt = tid - 64;
        KVM_PROBE_DECL(4)
        KVM_PROBE_START()
        int g = 0;
        for (int tt = 0;; ++tt) {
            const int id = tile_wait(tt);
            if (id < 0) break;
            const Tile T = tile_of(a, id);
            KVM_PROBE_LAP(3)
            if (!mbar_wait(bar(B_QFULL), tt & 1, abort_flag, a.status)) break;
            KVM_PROBE_LAP(0)
            if (half > 0) {
                for (int row = rt; row < 128; row += 64) {
                    const int64_t pos = T.q0 + row;
                    if (pos < a.N) {
                        if ((half & 7) == 0)
                            rope_row_vec(smem + OFF_Q + row * 128, row, pos, a.rope, half);
                        else
                            rope_row(smem + OFF_Q + row * 128, row, pos, a.rope, half);
                    }
                }
            }
            fence_proxy_async();
            mbar_arrive(bar(B_QREADY));
            bool ok = true;
            for (int j = 0; j < T.nblk; ++j, ++g) {
                const int s = g % NS;
                KVM_PROBE_LAP(2)
                if (!mbar_wait(bar(B_KFULL + s), (g / NS) & 1, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                KVM_PROBE_LAP(1)
                if (j >= T.nst && half > 0 && !a.k_rotated) {
                    const int64_t pos = T.ws + KB * (j - T.nst) + rt;
                    if (pos < a.N) {
                        if ((half & 7) == 0)
                            rope_row_vec(smem + OFF_K + s * KV_BYTES + rt * 128, rt, pos, a.rope, half);
                        else
                            rope_row(smem + OFF_K + s * KV_BYTES + rt * 128, rt, pos, a.rope, half);
                    }
                }
                fence_proxy_async();
                mbar_arrive(bar(B_KREADY + s));
            }
            if (!ok) break;
        }
        KVM_PROBE_LAP(2)
        if (rt == 0) KVM_PROBE_FLUSH(g_probe_attn, 8, 4)
    } else {
        // ------------------------------------------------------------ softmax
        const int row = tid - 128;                 // query row = TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tO = tmem + lane_base + TM_O;
        const float sc = a.scale_log2;
        KVM_PROBE_DECL(10)
        KVM_PROBE_START()
        int g = 0;
        bool ok = true;
        for (int tt = 0; ok; ++tt) {
            const int id = tile_wait(tt);
            if (id < 0) break;
            const Tile T = tile_of(a, id);
            const int64_t p = T.q0 + row;
            float m_used = -INFINITY, l = 0.0f;
            for (int j = 0; j < T.nblk; ++j) {
                const int gj = g + j, sb = gj & 1;
                KVM_PROBE_LAP(9)
                if (!mbar_wait(bar(B_SFULL + sb), (gj >> 1) & 1, abort_flag, a.status)) { ok = false; break; }
                KVM_PROBE_LAP(0)
#ifdef KVM_PROBE
                probe_acc[8] += 1;
#endif
                tc_fence_after();
                uint32_t v[2][32];
                tmem_ld32(tmem + lane_base + TM_S + sb * KB, v[0]);
                tmem_ld32(tmem + lane_base + TM_S + sb * KB + 32, v[1]);
                tmem_wait_ld();
                const bool is_state = j < T.nst;
                const int64_t key0 = is_state ? 0 : T.ws + KB * (j - T.nst);
                // columns < lim are valid keys for this query (a causal block may have none)
                int lim;
                if (is_state) {
                    lim = min(KB, T.n - KB * j);
                } else {
                    const int64_t d = p - key0 + 1;
                    lim = d < 0 ? 0 : (d < KB ? (int)d : KB);
                }
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                if (lim == KB) {
                    // a full block: every column is a valid key
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int x = 0; x < 32; ++x) mx[x & 3] = fmaxf(mx[x & 3], __uint_as_float(v[h][x]));
                } else {
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int x = 0; x < 32; ++x) {
                            const float val = h * 32 + x < lim ? __uint_as_float(v[h][x]) : -INFINITY;
                            v[h][x] = __float_as_uint(val);
                            mx[x & 3] = fmaxf(mx[x & 3], val);
                        }
                }
                const float mblk = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sc;
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
                KVM_PROBE_LAP(1)
                const float mneg = -m_used;
                uint32_t pk[32];
                float rs[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int x = 0; x < 32; x += 2) {
                        const float p0 = ex2(fmaf(__uint_as_float(v[h][x]), sc, mneg));
                        const float p1 = ex2(fmaf(__uint_as_float(v[h][x + 1]), sc, mneg));
                        rs[(x >> 1) & 3] += p0 + p1;
                        pk[(h * 32 + x) >> 1] = pack_bf16(p0, p1);
                    }
                l += (rs[0] + rs[1]) + (rs[2] + rs[3]);
                KVM_PROBE_LAP(4)
                // tensor-memory loads and stores are warp-wide (.sync.aligned): the whole
                // warp rescales when any of its rows must (the others scale by alpha = 1)
                if (__any_sync(0xffffffffu, rescale)) {
                    // O holds blocks < j: wait for their last PV, then scale it in place
                    if (!mbar_wait(bar(B_PVDONE + ((gj - 1) & 1)), ((gj - 1) >> 1) & 1, abort_flag, a.status)) { ok = false; break; }
                    tc_fence_after();
                    uint32_t o[32];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        tmem_ld32(tO + h * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
                        tmem_st32(tO + h * 32, o);
                    }
                    tmem_wait_st();
                }
                KVM_PROBE_LAP(3)
                // the P buffer was last read by the PV of block gj - 2
                if (gj >= 2 && !mbar_wait(bar(B_PVDONE + sb), ((gj - 2) >> 1) & 1, abort_flag, a.status)) { ok = false; break; }
                KVM_PROBE_LAP(2)
                uint8_t* prow = smem + OFF_P + sb * P_BYTES + row * 128;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                    *reinterpret_cast<uint4*>(prow + ((ch ^ (row & 7)) << 4)) =
                        make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
                fence_proxy_async();
                tc_fence_before();
                mbar_arrive(bar(B_PFULL + sb));
                KVM_PROBE_LAP(4)
            }
            if (!ok) break;
            // epilogue: O / l for this tile
            const int gl = g + T.nblk - 1;
            KVM_PROBE_LAP(9)
            if (!mbar_wait(bar(B_PVDONE + (gl & 1)), (gl >> 1) & 1, abort_flag, a.status)) { ok = false; break; }
            KVM_PROBE_LAP(5)
            tc_fence_after();
            const float il = 1.0f / l;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t o[32];
                tmem_ld32(tO + h * 32, o);
                tmem_wait_ld();
                if (p < a.N) {
                    uint4* dst = reinterpret_cast<uint4*>(a.out + ((int64_t)T.bh * a.N + p) * D) + h * 4;
#pragma unroll
                    for (int x = 0; x < 32; x += 8)
                        dst[x >> 3] = make_uint4(pack_bf16(__uint_as_float(o[x]) * il, __uint_as_float(o[x + 1]) * il),
                                                 pack_bf16(__uint_as_float(o[x + 2]) * il, __uint_as_float(o[x + 3]) * il),
                                                 pack_bf16(__uint_as_float(o[x + 4]) * il, __uint_as_float(o[x + 5]) * il),
                                                 pack_bf16(__uint_as_float(o[x + 6]) * il, __uint_as_float(o[x + 7]) * il));
                }
            }
            tc_fence_before();
            g += T.nblk;
            KVM_PROBE_LAP(6)
        }
        if (row == 0) KVM_PROBE_FLUSH(g_probe_attn, 12, 10)
    }

    tc_fence_before();
    __syncthreads();
#ifdef KVM_PROBE
    if (tid == 0) atomicAdd(&g_probe_attn[32 + (probe_sm & 31)], ~0ull);
#endif
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

KVM_PROBE_READOUT(kvm_probe_read_attn, g_probe_attn)

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

// 3-D bf16 map over [planes][rows][64] with a box_rows x 64 box, 128-byte swizzle.
bool make_tmap_bf16_3d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t planes, uint32_t box_rows) {
    using namespace tc;
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {64, rows, planes};
    cuuint64_t strides[2] = {64 * 2, rows * 64 * 2};
    cuuint32_t box[3] = {64, box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 3-D bf16 map over [planes][rows][row_elems] with a 64 x box_rows box, 128-byte swizzle
// (row_elems a multiple of 8: rows start on 16-byte boundaries).
bool make_tmap_bf16_rows(CUtensorMap* m, const void* base, uint64_t row_elems, uint64_t rows, uint64_t planes,
                         uint32_t box_rows) {
    using namespace tc;
    auto enc = get_encode();
    if (!enc || row_elems % 8) return false;
    cuuint64_t dims[3] = {row_elems, rows, planes};
    cuuint64_t strides[2] = {row_elems * 2, rows * row_elems * 2};
    cuuint32_t box[3] = {64, box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_tmap_f32_3d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t planes, uint32_t box_rows) {
    using namespace tc;
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[3] = {64, rows, planes};
    cuuint64_t strides[2] = {64 * 4, rows * 64 * 4};
    cuuint32_t box[3] = {32, box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, es,
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
    if (!make_tmap_bf16_3d(&mq, a.q, (uint64_t)a.N, BH, 128) || !make_tmap_bf16_3d(&mk, a.k_rot ? a.k_rot : a.k, (uint64_t)a.N, BH, KB) ||
        !make_tmap_bf16_3d(&mv, a.v, (uint64_t)a.N, BH, KB) ||
        !make_tmap_bf16_3d(&msk, a.snap_k, (uint64_t)a.M, planes_snap, KB) ||
        !make_tmap_bf16_3d(&msv, a.snap_v, (uint64_t)a.M, planes_snap, KB))
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
    t.k_rotated = a.k_rot != nullptr;
    t.tile_ctr = a.tile_ctr;
    t.n_ranges = a.n_ranges < AttnArgs::MAX_RANGES ? a.n_ranges : AttnArgs::MAX_RANGES;
    for (int r = 0; r < AttnArgs::MAX_RANGES; ++r) {
        const int e = r < t.n_ranges ? a.range_end[r] : t.ntiles;
        t.range_end[r] = e < t.ntiles ? e : t.ntiles;
    }
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
    static int per_sm = 0;
    if (per_sm == 0) {
        cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
        // Two CTAs per SM fit (2 x 97 KB shared memory, 2 x 256 x 128 registers, 2 x 256
        // TMEM columns), but the occupancy calculator reports one for this kernel.  CTAs
        // of the persistent grid never wait on each other, so a grid of two per SM is
        // correct whether or not both are resident.
        per_sm = 2;
#ifdef KVM_PROBE
        {
            int dev = 0, smem_sm = 0, resv = 0, regs_sm = 0, occ = -1;
            cudaGetDevice(&dev);
            cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
            cudaDeviceGetAttribute(&resv, cudaDevAttrReservedSharedMemoryPerBlock, dev);
            cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev);
            cudaError_t oe = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, attn_tc_kernel, 256, SMEM_BYTES);
            cudaFuncAttributes fa;
            cudaFuncGetAttributes(&fa, attn_tc_kernel);
            for (int sz : {0, 16384, 49152, 65536, 81920, 99584}) {
                int o2 = -1;
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o2, attn_tc_kernel, 256, sz);
                int o3 = -1;
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o3, attn_tc_kernel, 128, sz);
                fprintf(stderr, "[probe] dyn smem %d -> occupancy %d (256 thr) %d (128 thr)\n", sz, o2, o3);
            }
            fprintf(stderr, "[probe] attn occupancy %d (err %d %s) smem/SM %d reserved/block %d regs/SM %d "
                    "kernel regs %d static smem %zu dyn %d maxdyn %d\n", occ, (int)oe, cudaGetErrorString(oe),
                    smem_sm, resv, regs_sm, fa.numRegs, fa.sharedSizeBytes, SMEM_BYTES, fa.maxDynamicSharedSizeBytes);
        }
#endif
    }
    int grid = a.grid > 0 ? a.grid : per_sm * nsm;
    if (!a.tile_ctr && grid > t.ntiles) grid = t.ntiles;
    attn_tc_kernel<<<grid, 256, SMEM_BYTES, s>>>(mq, mk, mv, msk, msv, t);
    return cudaGetLastError();
}

}  // namespace kvm
