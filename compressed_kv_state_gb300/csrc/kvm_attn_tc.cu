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
// Persistent CTAs (one per SM, 384 threads, 225 KB shared memory, all 512
// tensor-memory columns) hold two tile slots.  Each slot has its own roles, so
// the tensor core runs one slot's QK^T and PV while the other slot's softmax
// works; tiles are taken statically strided or claimed from counters shared by
// several launches.  Per slot:
//   producer warp (0, 1)   claims the slot's tiles, loads Q and the K/V blocks
//                          by TMA (3 stages of 128 keys)
//   MMA warp (2, 3)        one thread issues S = Q K^T (N = 128) into the slot's
//                          128-column S, then O += P V with P read from tensor
//                          memory (the A-from-tensor-memory form); the next
//                          block's QK^T follows that PV in issue order
//   softmax warps (4-7,    thread i owns query row i (= TMEM lane i): rotates
//   8-11)                  its row of the Q tile, then per block a max pass
//                          and an exponent pass over the S row (packed fp32,
//                          three-input max), lazy rescaling of O (only when the
//                          running maximum grows by more than 2^8), P written
//                          back as bf16 pairs over the first 64 S columns;
//                          finally O / l to the output.
// All mbarrier waits are bounded (about two seconds); on expiry the CTA
// raises the device status word, lets its issued copies and MMAs land, and
// exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>

#include "kvm_internal.cuh"
#include "tc_primitives.cuh"

namespace kvm {
namespace tc {

#ifdef KVM_PROBE
static __device__ unsigned long long g_probe_attn[64];
#endif

struct TcArgs {
    int64_t N;
    int BH, C, W, M, r;
    int tiles_per_head, ntiles;
    int* tile_ctr;   // dynamic claiming: one counter per range (nullptr: static striding)
    int n_ranges;
    int range_end[AttnArgs::MAX_RANGES];
    int snap_events;
    const Sched* sched;
    const float2* rope;
    float scale_log2;
    __nv_bfloat16* out;
    int* status;
    int q_prerot;    // queries come rotated: no RoPE in the kernel, the MMA waits for the copy
    float* lse;      // optional: log2-sum-exp per query
    int split;       // Q and window-K tiles as two 64-byte halves: rotated dims [0, 32) from
                     // the compact q_rot / k_rot rows, dims [32, 64) from q / k
};

struct Tile {
    int bh, e, n, nst, nwin, nblk;
    int64_t q0, ws;
};

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

// Two query tiles in flight per CTA (one CTA per SM), each with its own
// producer, MMA issuer and softmax warpgroup; while one tile's softmax runs,
// the tensor core works on the other tile's QK^T and PV.
constexpr int NSLOT = 2;              // query tiles in flight per CTA
constexpr int NS = 3;                 // K/V stages per tile slot
constexpr int KB = 128;               // keys per block
constexpr int Q_BYTES = 128 * 128;    // Q tile [128 x 64] bf16
constexpr int KV_BYTES = KB * 128;    // K or V block [128 x 64] bf16
constexpr int OFF_Q = 0;                               // [NSLOT] Q tiles
constexpr int OFF_K = OFF_Q + NSLOT * Q_BYTES;         // [NSLOT][NS] K blocks
constexpr int OFF_V = OFF_K + NSLOT * NS * KV_BYTES;   // [NSLOT][NS] V blocks
constexpr int OFF_BAR = OFF_V + NSLOT * NS * KV_BYTES;
constexpr int SMEM_BYTES = OFF_BAR + 512 + 1024;       // 225.5 KB with alignment slack
constexpr int TMEM_COLS = 512;                         // per slot (256 columns): S (128),
                                                       // O (64), P (64: bf16 key pairs)
constexpr int NTHREADS = 384;
// Register split (the block is launched with 168 registers a thread, 64512 in
// all): the producer / MMA warpgroup drops to 64, the two softmax warpgroups rise
// to 216, which keeps a whole 128-column S row in registers: 4 * 32 * 64 +
// 8 * 32 * 216 = 63488 <= 64512.
constexpr int REGS_LOW = 64, REGS_HIGH = 216;
constexpr float TAU = 8.0f;  // lazy-rescale threshold (log2 units)

// per-slot barrier indices
enum {
    B_QFULL = 0,                 // TMA Q landed
    B_QREADY = 1,                // Q rotated (128 arrivals)
    B_QEMPTY = 2,                // last QK of the tile done
    B_KFULL = 3,                 // [NS] TMA K landed
    B_VFULL = B_KFULL + NS,      // [NS] TMA V landed
    B_KVEMPTY = B_VFULL + NS,    // [NS] PV of the stage done
    B_SFULL = B_KVEMPTY + NS,    // QK done
    B_SFREE = B_SFULL + 1,       // S read into registers by the softmax (128 arrivals)
    B_PFULL = B_SFREE + 1,       // P written to tensor memory, O rescaled (128 arrivals)
    B_PVDONE = B_PFULL + 1,      // PV done
    B_FINAL = B_PVDONE + 1,      // MMA drain
    B_TILE = B_FINAL + 1,        // [4] tile number of turn k published (ring of 4)
    NBAR_SLOT = B_TILE + 4
};

__device__ __forceinline__ Tile tile_of2(const TcArgs& a, int id) {
    Tile t;
    t.bh = id % a.BH;
    t.q0 = (int64_t)(id / a.BH) * 128;
    const int64_t c = t.q0 / a.C, Wc = a.W / a.C;
    t.e = (int)(c - Wc - 1);
    t.n = t.e >= 0 ? a.sched[t.e].n_after : 0;
    if (t.n > 0 && !kvm_check(t.e < a.snap_events && t.n <= a.M, a.status)) t.n = 0;
    t.ws = c - Wc > 0 ? (c - Wc) * a.C : 0;
    t.nst = (t.n + KB - 1) / KB;
    t.nwin = (int)((t.q0 + 128 - t.ws + KB - 1) / KB);
    t.nblk = t.nst + t.nwin;
    return t;
}

// The tile a slot processes in its k-th turn, or -1 when it is done.  Dynamic:
// one atomicAdd per claim on the first range (from *range on) not exhausted.
// Static: turn k of slot s is the CTA's turn 2k + s.
__device__ __forceinline__ int next_tile2(const TcArgs& a, int slot, int k, int* range) {
    if (a.tile_ctr) {
        for (; *range < a.n_ranges; ++*range) {
            const int r = *range;
            const int lo = r > 0 ? a.range_end[r - 1] : 0;
            const int id = lo + atomicAdd(a.tile_ctr + r, 1);
            if (id < a.range_end[r]) return id;
        }
        return -1;
    }
    const int64_t id = blockIdx.x + (int64_t)(2 * k + slot) * gridDim.x;
    return id < a.ntiles ? (int)id : -1;
}

// wait for a phase without the abort shortcut (drains after an abort), bounded
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try(bar, parity) && clock64() - t0 < (1ll << 28)) {
    }
}

__global__ void __launch_bounds__(NTHREADS, 1)
    attn_tc2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_sk,
                    const __grid_constant__ CUtensorMap tm_sv, const __grid_constant__ CUtensorMap tm_qh,
                    const __grid_constant__ CUtensorMap tm_kh, const TcArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NSLOT * NBAR_SLOT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* tile_ring = reinterpret_cast<volatile int*>(tmem_slot + 2);  // [NSLOT][4]
    auto bar = [&](int slot, int i) { return smem_u32(bars + slot * NBAR_SLOT + i); };
    // The producer of a slot publishes the tile of its turn k in ring entry k % 4; the
    // other roles read it after that entry's barrier.  An entry is rewritten four turns
    // later: the producer claims turn k only after the last QK MMA of turn k - 1, which
    // follows the Q rotation of turn k - 1 and the softmax of turn k - 2's last block.
    auto tile_wait = [&](int slot, int k) -> int {
        if (!mbar_wait(bar(slot, B_TILE + (k & 3)), (k >> 2) & 1, abort_flag, a.status)) return -1;
        return tile_ring[slot * 4 + (k & 3)];
    };

    if (tid == 0) {
        for (int s = 0; s < NSLOT; ++s) {
            mbar_init(bar(s, B_QFULL), 1);
            mbar_init(bar(s, B_QREADY), 128);
            mbar_init(bar(s, B_QEMPTY), 1);
            for (int i = 0; i < NS; ++i) {
                mbar_init(bar(s, B_KFULL + i), 1);
                mbar_init(bar(s, B_VFULL + i), 1);
                mbar_init(bar(s, B_KVEMPTY + i), 1);
            }
            mbar_init(bar(s, B_SFULL), 1);
            mbar_init(bar(s, B_SFREE), 128);
            mbar_init(bar(s, B_PFULL), 128);
            mbar_init(bar(s, B_PVDONE), 1);
            mbar_init(bar(s, B_FINAL), 1);
            for (int i = 0; i < 4; ++i) mbar_init(bar(s, B_TILE + i), 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async();
    }
    if (warp == 2) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sbase = smem_u32(smem);
    const int half = a.r / 2;
    if (warp < 4)
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_LOW));
    else
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REGS_HIGH));

    if (warp < 2) {
        // ------------------------------------------------------------ producer
        const int slot = warp;
        int last_g = -1;  // last block whose K/V copies were issued
        if (lane == 0) {
            int g = 0, range = 0;
            KVM_PROBE_DECL(4)
            KVM_PROBE_START()
            for (int k = 0;; ++k) {
                // the next tile is picked and published before its query buffer is free
                // (consumers are at most two tiles behind: the ring holds four)
                const int id = next_tile2(a, slot, k, &range);
                tile_ring[slot * 4 + (k & 3)] = id;
                mbar_arrive(bar(slot, B_TILE + (k & 3)));
                if (id < 0) break;
                const Tile T = tile_of2(a, id);
                if (k >= 1 && !mbar_wait(bar(slot, B_QEMPTY), (k - 1) & 1, abort_flag, a.status)) break;
                KVM_PROBE_LAP(2)
                mbar_expect_tx(bar(slot, B_QFULL), Q_BYTES);
                if (a.split) {  // rotated half, then dims [32, 64) of the unrotated row
                    tma_load_3d(sbase + OFF_Q + slot * Q_BYTES, &tm_q, 0, (int)T.q0, T.bh, bar(slot, B_QFULL));
                    tma_load_3d(sbase + OFF_Q + slot * Q_BYTES + Q_BYTES / 2, &tm_qh, 32, (int)T.q0, T.bh,
                                bar(slot, B_QFULL));
                } else {
                    tma_load_3d(sbase + OFF_Q + slot * Q_BYTES, &tm_q, 0, (int)T.q0, T.bh, bar(slot, B_QFULL));
                }
                bool ok = true;
                for (int j = 0; j < T.nblk; ++j, ++g) {
                    const int st = g % NS;
                    KVM_PROBE_LAP(1)
                    if (g >= NS && !mbar_wait(bar(slot, B_KVEMPTY + st), ((g / NS) - 1) & 1, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    KVM_PROBE_LAP(0)
                    const uint32_t dk = sbase + OFF_K + (slot * NS + st) * KV_BYTES;
                    const uint32_t dv = sbase + OFF_V + (slot * NS + st) * KV_BYTES;
                    mbar_expect_tx(bar(slot, B_KFULL + st), KV_BYTES);
                    mbar_expect_tx(bar(slot, B_VFULL + st), KV_BYTES);
                    if (j < T.nst) {
                        const int plane = T.bh * a.snap_events + T.e;
                        tma_load_3d(dk, &tm_sk, 0, KB * j, plane, bar(slot, B_KFULL + st));
                        tma_load_3d(dv, &tm_sv, 0, KB * j, plane, bar(slot, B_VFULL + st));
                    } else {
                        const int key0 = (int)(T.ws + KB * (j - T.nst));
                        tma_load_3d(dk, &tm_k, 0, key0, T.bh, bar(slot, B_KFULL + st));
                        if (a.split) tma_load_3d(dk + KV_BYTES / 2, &tm_kh, 32, key0, T.bh, bar(slot, B_KFULL + st));
                        tma_load_3d(dv, &tm_v, 0, key0, T.bh, bar(slot, B_VFULL + st));
                    }
                    last_g = g;
                }
                if (!ok) break;
            }
            KVM_PROBE_LAP(1)
            if (slot == 0) KVM_PROBE_FLUSH(g_probe_attn, 0, 3)
            // after an abort: the copies issued last on every stage land before exit
            if (*abort_flag)
                for (int gg = last_g; gg >= 0 && gg > last_g - NS; --gg) {
                    drain_wait(bar(slot, B_KFULL + gg % NS), (gg / NS) & 1);
                    drain_wait(bar(slot, B_VFULL + gg % NS), (gg / NS) & 1);
                }
        }
    } else if (warp < 4) {
        // ---------------------------------------------------------- MMA issuer
        const int slot = warp - 2;
        if (lane == 0) {
            const uint32_t idesc_qk = idesc_bf16(128, KB, 0, 0);
            const uint32_t idesc_pv = idesc_bf16(128, 64, 0, 1);
            const int ks_state = min(a.r / 16, 3);
            const uint32_t tS = tmem + 256 * slot, tO = tS + 128, tP = tS + 192;
            const uint32_t sQ = sbase + OFF_Q + slot * Q_BYTES;
            // shared-memory descriptors of the slot's Q tile and of its first K and V stage
            const uint64_t dq0 = sdesc_sw128(sQ, 16, 1024);
            const uint64_t dk0 = sdesc_sw128(sbase + OFF_K + slot * NS * KV_BYTES, 16, 1024);
            const uint64_t dv0 = sdesc_sw128(sbase + OFF_V + slot * NS * KV_BYTES, KV_BYTES, 1024);
            // the same tiles as 64-byte-swizzled halves (split Q and window K)
            const uint64_t dq64 = sdesc_sw64(sQ);
            const uint64_t dk64 = sdesc_sw64(sbase + OFF_K + slot * NS * KV_BYTES);
            int g = 0;
            bool ok = true;
            KVM_PROBE_DECL(8)
            KVM_PROBE_START()
            // S = Q K^T of block gb (state blocks: the non-rotary dims only; the state keys
            // are zero on the rotary dims), once the softmax has read block gb - 1's S
            auto issue_qk = [&](int gb, bool state) -> bool {
                const int st = gb % NS;
                if (gb > 0 && !mbar_wait(bar(slot, B_SFREE), (gb - 1) & 1, abort_flag, a.status)) return false;
                if (!mbar_wait(bar(slot, B_KFULL + st), (gb / NS) & 1, abort_flag, a.status)) return false;
                KVM_PROBE_LAP(1)
                tc_fence_after();
                // descriptors: the address field is the byte address / 16, so a K-step of
                // 32 bytes adds 2 and a stage adds KV_BYTES / 16
                const uint64_t dk = dk0 + (uint64_t)(st * (KV_BYTES >> 4));
                const int ks0 = state ? ks_state : 0;
                if (a.split) {
                    // 64-byte halves: K-steps 0, 1 in the rotated half, 2, 3 in the other
                    // (state keys: the 128-byte-swizzled rows of the snapshot, K-steps 2, 3)
                    const uint64_t dks64 = dk64 + (uint64_t)(st * (KV_BYTES >> 4));
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        if (ks < ks0) continue;
                        const uint64_t ad = dq64 + (uint64_t)((ks >> 1) * (Q_BYTES / 2 >> 4) + 2 * (ks & 1));
                        const uint64_t bd = state ? dk + 2 * ks
                                                  : dks64 + (uint64_t)((ks >> 1) * (KV_BYTES / 2 >> 4) + 2 * (ks & 1));
                        mma_bf16_ss(tS, ad, bd, idesc_qk, ks > ks0);
                    }
                } else {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        if (ks >= ks0) mma_bf16_ss(tS, dq0 + 2 * ks, dk + 2 * ks, idesc_qk, ks > ks0);
                }
                mma_commit(bar(slot, B_SFULL));
                KVM_PROBE_LAP(2)
                return true;
            };
            for (int k = 0; ok; ++k) {
                const int id = tile_wait(slot, k);
                if (id < 0) break;
                const Tile T = tile_of2(a, id);
                KVM_PROBE_LAP(6)
                if (!mbar_wait(bar(slot, a.q_prerot ? B_QFULL : B_QREADY), k & 1, abort_flag, a.status)) break;
                KVM_PROBE_LAP(0)
                tc_fence_after();
                if (!issue_qk(g, T.nst > 0)) break;
                // the query tile is free once the tile's last QK^T completes: the next
                // tile's query loads while this tile's last blocks run
                if (T.nblk == 1) mma_commit(bar(slot, B_QEMPTY));
                for (int j = 0; j < T.nblk; ++j) {
                    const int gj = g + j, st = gj % NS;
                    // the next block's QK^T overlaps this block's softmax
                    if (j + 1 < T.nblk) {
                        if (!issue_qk(gj + 1, j + 1 < T.nst)) { ok = false; break; }
                        if (j + 2 == T.nblk) mma_commit(bar(slot, B_QEMPTY));
                    }
                    if (!mbar_wait(bar(slot, B_PFULL), gj & 1, abort_flag, a.status)) { ok = false; break; }
                    KVM_PROBE_LAP(3)
                    if (!mbar_wait(bar(slot, B_VFULL + st), (gj / NS) & 1, abort_flag, a.status)) { ok = false; break; }
                    KVM_PROBE_LAP(4)
                    tc_fence_after();
                    // O += P V: P (bf16, two keys per column) from tensor memory, V from shared
                    const uint64_t dv = dv0 + (uint64_t)(st * (KV_BYTES >> 4));
#pragma unroll
                    for (int ks = 0; ks < KB / 16; ++ks)
                        mma_bf16_ts(tO, tP + 8 * ks, dv + 128 * ks, idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
                    mma_commit(bar(slot, B_PVDONE));
                    mma_commit(bar(slot, B_KVEMPTY + st));
                    KVM_PROBE_LAP(5)
#ifdef KVM_PROBE
                    probe_acc[7] += 1;
#endif
                }
                g += T.nblk;
            }
            if (slot == 0) KVM_PROBE_FLUSH(g_probe_attn, 8, 8)
            // every MMA this thread issued completes before the tensor memory is released
            mma_commit(bar(slot, B_FINAL));
            drain_wait(bar(slot, B_FINAL), 0);
        }
    } else {
        // ------------------------------------------------------------ softmax
        const int slot = (warp - 4) >> 2;
        const int row = tid - 128 - 128 * slot;                // query row = TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_base + 256 * slot, tO = tS + 128, tP = tS + 192;
        uint8_t* qrow = smem + OFF_Q + slot * Q_BYTES + row * 128;
        const float sc = a.scale_log2;
        const float2 sc2 = make_float2(sc, sc);
        int g = 0;
        bool ok = true;
        KVM_PROBE_DECL(10)
        KVM_PROBE_START()
        for (int k = 0; ok; ++k) {
            const int id = tile_wait(slot, k);
            if (id < 0) break;
            const Tile T = tile_of2(a, id);
            const int64_t p = T.q0 + row;
            // RoPE of this thread's query row, then hand the tile to the MMA (nothing to
            // do when the queries come rotated: the MMA waits for their copy itself)
            if (!a.q_prerot) {
                if (!mbar_wait(bar(slot, B_QFULL), k & 1, abort_flag, a.status)) break;
                KVM_PROBE_LAP(0)
                if (half > 0 && p < a.N) {
                    if ((half & 7) == 0)
                        rope_row_vec(qrow, row, p, a.rope, half);
                    else
                        rope_row(qrow, row, p, a.rope, half);
                }
                fence_proxy_async();
                mbar_arrive(bar(slot, B_QREADY));
            }
            KVM_PROBE_LAP(1)
            float m_used = -INFINITY, l = 0.0f;
            for (int j = 0; j < T.nblk; ++j) {
                const int gj = g + j;
                if (!mbar_wait(bar(slot, B_SFULL), gj & 1, abort_flag, a.status)) { ok = false; break; }
                KVM_PROBE_LAP(2)
#ifdef KVM_PROBE
                probe_acc[9] += 1;
#endif
                tc_fence_after();
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
                // the whole S row of this block in registers (one tensor-memory round trip)
                uint32_t v[KB / 32][32];
#pragma unroll
                for (int h = 0; h < KB / 32; ++h) tmem_ld32(tS + 32 * h, v[h]);
                tmem_wait_ld();
                // S is in registers: the next block's QK^T may overwrite it
                tc_fence_before();
                mbar_arrive(bar(slot, B_SFREE));
                if (lim < KB) {
#pragma unroll
                    for (int h = 0; h < KB / 32; ++h)
#pragma unroll
                        for (int x = 0; x < 32; ++x)
                            if (32 * h + x >= lim) v[h][x] = __float_as_uint(-INFINITY);
                }
                // the block's row maximum
                float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                for (int h = 0; h < KB / 32; ++h)
#pragma unroll
                    for (int x = 0; x < 32; x += 4) {
                        mx0 = fmax3(mx0, __uint_as_float(v[h][x]), __uint_as_float(v[h][x + 1]));
                        mx1 = fmax3(mx1, __uint_as_float(v[h][x + 2]), __uint_as_float(v[h][x + 3]));
                    }
                const float mblk = fmaxf(mx0, mx1) * sc;
                KVM_PROBE_LAP(3)
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
                // the previous block's PV has read P and updated O (it ran while this
                // block's S was loaded and reduced)
                if (gj > 0 && !mbar_wait(bar(slot, B_PVDONE), (gj - 1) & 1, abort_flag, a.status)) { ok = false; break; }
                tc_fence_after();
                // tensor-memory loads and stores are warp-wide (.sync.aligned): the whole
                // warp rescales when any of its rows must (the others scale by alpha = 1)
                if (__any_sync(0xffffffffu, rescale)) {
                    uint32_t o[32];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        tmem_ld32(tO + h * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
                        tmem_st32(tO + h * 32, o);
                    }
                }
                // p = 2^(s * scale - m), row sum, P as bf16 key pairs into the P columns
                const float2 mneg = make_float2(-m_used, -m_used);
                float2 rs[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                make_float2(0.f, 0.f)};
#pragma unroll
                for (int h = 0; h < KB / 32; ++h) {
                    uint32_t pk[16];
#pragma unroll
                    for (int x = 0; x < 32; x += 2) {
                        const float2 s2 = make_float2(__uint_as_float(v[h][x]), __uint_as_float(v[h][x + 1]));
                        const float2 t2 = __ffma2_rn(s2, sc2, mneg);
                        const float2 e2 = make_float2(ex2(t2.x), ex2(t2.y));
                        rs[(x >> 1) & 3] = __fadd2_rn(rs[(x >> 1) & 3], e2);
                        pk[x >> 1] = pack_bf16(e2.x, e2.y);
                    }
                    tmem_st16(tP + 16 * h, pk);
                }
                tmem_wait_st();
                KVM_PROBE_LAP(4)
                l += ((rs[0].x + rs[0].y) + (rs[1].x + rs[1].y)) + ((rs[2].x + rs[2].y) + (rs[3].x + rs[3].y));
                tc_fence_before();
                mbar_arrive(bar(slot, B_PFULL));
                KVM_PROBE_LAP(5)
            }
            if (!ok) break;
            // epilogue: O / l for this tile
            const int gl = g + T.nblk - 1;
            if (!mbar_wait(bar(slot, B_PVDONE), gl & 1, abort_flag, a.status)) { ok = false; break; }
            KVM_PROBE_LAP(6)
            tc_fence_after();
            const float il = 1.0f / l;
            if (a.lse && p < a.N) a.lse[(int64_t)T.bh * a.N + p] = m_used + log2f(l);
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
            KVM_PROBE_LAP(7)
        }
        if (slot == 0 && row == 0) KVM_PROBE_FLUSH(g_probe_attn, 16, 10)
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
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

// 3-D bf16 map over [planes][rows][row_elems] with a 32 x box_rows box, 64-byte swizzle
// (row_elems 32 or 64; a box of dims [32, 64) starts at x = 32).
static bool make_tmap_bf16_half(CUtensorMap* m, const void* base, uint64_t row_elems, uint64_t rows,
                                uint64_t planes, uint32_t box_rows) {
    using namespace tc;
    auto enc = get_encode();
    if (!enc || (row_elems != 32 && row_elems != 64)) return false;
    cuuint64_t dims[3] = {row_elems, rows, planes};
    cuuint64_t strides[2] = {row_elems * 2, rows * row_elems * 2};
    cuuint32_t box[3] = {32, box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool attn_tc_supported(const AttnArgs& a, bool bf16) {
    return bf16 && a.C % 128 == 0 && a.N > 0;
}

cudaError_t launch_attn_tc(const AttnArgs& a, int* status, cudaStream_t s) {
    using namespace tc;
    CUtensorMap mq, mk, mv, msk, msv, mqh, mkh;
    const uint64_t BH = (uint64_t)a.BH;
    const uint64_t planes_snap = BH * (uint64_t)(a.snap_events > 0 ? a.snap_events : 1);
    // window keys must come rotated at their own positions when the layer has rotary dims
    if (a.r > 0 && !a.k_rot) return cudaErrorInvalidValue;
    // compact rotated rows (r = 32): Q and window-K tiles in two 64-byte halves
    const bool split = a.rot_compact != 0;
    if (split && (a.r != 32 || !a.q_rot)) return cudaErrorInvalidValue;
    bool maps_ok;
    if (split)
        maps_ok = make_tmap_bf16_half(&mq, a.q_rot, 32, (uint64_t)a.N, BH, 128) &&
                  make_tmap_bf16_half(&mqh, a.q, 64, (uint64_t)a.N, BH, 128) &&
                  make_tmap_bf16_half(&mk, a.k_rot, 32, (uint64_t)a.N, BH, KB) &&
                  make_tmap_bf16_half(&mkh, a.k, 64, (uint64_t)a.N, BH, KB);
    else
        maps_ok = make_tmap_bf16_3d(&mq, a.q_rot ? a.q_rot : a.q, (uint64_t)a.N, BH, 128) &&
                  make_tmap_bf16_3d(&mk, a.k_rot ? a.k_rot : a.k, (uint64_t)a.N, BH, KB);
    if (!split) {  // unused by the kernel: any valid map
        mqh = mq;
        mkh = mk;
    }
    if (!maps_ok || !make_tmap_bf16_3d(&mv, a.v, (uint64_t)a.N, BH, KB) ||
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
    t.q_prerot = a.q_rot != nullptr || a.r == 0;
    t.lse = a.lse;
    t.split = split ? 1 : 0;
    static int nsm = 0;
    if (nsm == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        cudaFuncSetAttribute(attn_tc2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    }
    // persistent: one CTA per SM (two query tiles in flight in each); a.grid, when
    // given, is the number of CTAs for the SM partition the launch runs on
    int grid = a.grid > 0 ? a.grid : nsm;
    if (!a.tile_ctr && grid > (t.ntiles + 1) / 2) grid = (t.ntiles + 1) / 2;
    attn_tc2_kernel<<<grid, NTHREADS, SMEM_BYTES, s>>>(mq, mk, mv, msk, msv, mqh, mkh, t);
    return cudaGetLastError();
}

}  // namespace kvm
