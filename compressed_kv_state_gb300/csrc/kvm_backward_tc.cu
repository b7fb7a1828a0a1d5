// Backward of the KVM prefill on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// "Key-Value Means" (gist.science technical summary), Methodology and Core mechanism
// 4: the gradient of the one softmax over the state's read view and the RoPE window,
// at the forward's fold decisions.  This file holds the five attention products of the
// backward for bf16 layers whose chunks are multiples of 128 (the forward's
// tensor-core attention then kept every query's log2-sum-exp):
//   S = Q K^T, dP = dO V^T, P = 2^(S * scale_log2 - lse), dS = P (dP - dout . out),
//   dV = P^T dO, dK = dS^T Q, dQ += dS K.
// The read rows' gradients per event and slot, the window keys' gradients (in rotated
// coordinates) and dq (rotated back) leave the tile; the slot sweep and the rotation of
// dk back run in kvm_backward.cu.
//
// One CTA per (row, 128-query tile); 320 threads:
//   warp 0        producer: the tile's Q and dO, then its key blocks (128 keys: the
//                 read rows of its chunk's state, then its window) by TMA, 2 stages
//   warp 1        one thread issues the MMAs: S and dP (A and B K-major) into tensor
//                 memory; once P and dS are in shared memory, the next block's S and dP,
//                 then dV = P^T dO and dK = dS^T Q (A MN-major: keys run along the rows
//                 of P and dS) and dQ += dS K
//   warps 2-9     two warpgroups; thread i of warpgroup g owns query row i (= tensor-
//                 memory lane i) and keys [64g, 64g + 64) of each block: P and dS of that
//                 part of its row in registers (while the previous block's products run);
//                 then, as key row i, dims [32g, 32g + 32) of the previous block's dK and
//                 dV rows to the gradient arrays (vector reductions through a per-warp
//                 staging area); then P and dS as bf16 into 64-key 128-byte-swizzled half
//                 tile g; at the end dims [32g, 32g + 32) of its dQ row, scaled and
//                 rotated back, to dq.
// Tensor memory (512 columns): S 128, dP 128, dQ 64, dK 64, dV 64.  All mbarrier waits are
// bounded; on expiry the CTA raises the status word, lets its copies and MMAs land, exits.
#include <cuda.h>
#include <cuda_bf16.h>

#include "kvm_internal.cuh"
#include "tc_primitives.cuh"

namespace kvm {
namespace bwt {

using namespace tc;

constexpr int TQ = 128;          // queries per tile
constexpr int KB = 128;          // keys per block
constexpr int NS = 2;            // K/V stages
constexpr int TILE = 128 * 128;  // bytes of a [128][64] bf16 tile (128-byte swizzled rows)
constexpr int OFF_Q = 0;
constexpr int OFF_DO = OFF_Q + TILE;
constexpr int OFF_K = OFF_DO + TILE;        // [NS]
constexpr int OFF_V = OFF_K + NS * TILE;    // [NS]
constexpr int OFF_P = OFF_V + NS * TILE;    // two halves: keys [0, 64) and [64, 128), [128 queries][128 B]
constexpr int OFF_DS = OFF_P + 2 * TILE;    // the same for dS
constexpr int OFF_STG = OFF_DS + 2 * TILE;  // per softmax-gradient warp: [32 rows][32 floats]
constexpr int STG_FLOATS = 32 * 32;
constexpr int OFF_BAR = OFF_STG + 8 * STG_FLOATS * 4;  // 192 KB
constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;
constexpr int NTHREADS = 320;
constexpr int NSM = 256;  // softmax-gradient threads (two warpgroups)
constexpr int T_S = 0, T_DP = 128, T_DQ = 256, T_DK = 320, T_DV = 384;  // tensor-memory columns

enum {
    B_QFULL = 0,              // Q and dO landed
    B_KFULL = 1,              // [NS]
    B_VFULL = B_KFULL + NS,   // [NS]
    B_KVEMPTY = B_VFULL + NS, // [NS] the stage's last MMA done
    B_SPD = B_KVEMPTY + NS,   // S and dP of the block in tensor memory
    B_PDS,                    // S and dP read, P and dS in shared memory (256 arrivals)
    B_MMA2,                   // dV, dK, dQ MMAs of the block done
    B_DKVFREE,                // dK and dV of the block read out (256 arrivals)
    B_FINAL,                  // MMA drain
    NBAR
};

__device__ __forceinline__ uint32_t packbf2(float x, float y) {
    __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    return *reinterpret_cast<uint32_t*>(&h);
}

// bounded wait with no abort shortcut (drains after an abort)
__device__ __forceinline__ void drain(uint32_t bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try(bar, parity) && clock64() - t0 < (1ll << 28)) {
    }
}

__global__ void __launch_bounds__(NTHREADS, 1)
    bwd_tc5_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_sk, const __grid_constant__ CUtensorMap tm_sv,
                   const BackwardArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + NBAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    auto bar = [&](int i) { return smem_u32(bars + i); };
    const uint32_t sbase = smem_u32(sm);

    const int tiles = (int)((a.N + TQ - 1) / TQ);
    const int bh = blockIdx.x / tiles;
    const int64_t q0 = (int64_t)(blockIdx.x % tiles) * TQ;
    const int nq = (int)(a.N - q0 < TQ ? a.N - q0 : TQ);
    const int Wc = a.W / a.C;
    const int64_t c = q0 / a.C, e = c - Wc - 1, ws = c - Wc > 0 ? (c - Wc) * a.C : 0;
    int n = e >= 0 ? a.sched[e].n_after : 0;
    if (n > a.M) n = a.M;
    const int nbs = (n + KB - 1) / KB;
    const int nbw = (int)((q0 + nq - ws + KB - 1) / KB);
    const int nblk = nbs + nbw;
    const int64_t row = (int64_t)bh * a.N;

    if (tid == 0) {
        mbar_init(bar(B_QFULL), 1);
        for (int i = 0; i < NS; ++i) {
            mbar_init(bar(B_KFULL + i), 1);
            mbar_init(bar(B_VFULL + i), 1);
            mbar_init(bar(B_KVEMPTY + i), 1);
        }
        mbar_init(bar(B_SPD), 1);
        mbar_init(bar(B_PDS), NSM);
        mbar_init(bar(B_MMA2), 1);
        mbar_init(bar(B_DKVFREE), NSM);
        mbar_init(bar(B_FINAL), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            mbar_expect_tx(bar(B_QFULL), 2 * TILE);
            tma_load_3d(sbase + OFF_Q, &tm_q, 0, (int)q0, bh, bar(B_QFULL));
            tma_load_3d(sbase + OFF_DO, &tm_do, 0, (int)q0, bh, bar(B_QFULL));
            int last = -1;
            for (int j = 0; j < nblk; ++j) {
                const int st = j % NS;
                if (j >= NS && !mbar_wait(bar(B_KVEMPTY + st), ((j / NS) - 1) & 1, abort_flag, a.status)) break;
                const uint32_t dk = sbase + OFF_K + st * TILE, dv = sbase + OFF_V + st * TILE;
                mbar_expect_tx(bar(B_KFULL + st), TILE);
                mbar_expect_tx(bar(B_VFULL + st), TILE);
                if (j < nbs) {
                    const int plane = bh * a.snap_events + (int)e;
                    tma_load_3d(dk, &tm_sk, 0, KB * j, plane, bar(B_KFULL + st));
                    tma_load_3d(dv, &tm_sv, 0, KB * j, plane, bar(B_VFULL + st));
                } else {
                    const int key0 = (int)(ws + KB * (j - nbs));
                    tma_load_3d(dk, &tm_k, 0, key0, bh, bar(B_KFULL + st));
                    tma_load_3d(dv, &tm_v, 0, key0, bh, bar(B_VFULL + st));
                }
                last = j;
            }
            drain(bar(B_QFULL), 0);
            if (*abort_flag)  // the copies issued last on every stage land before exit
                for (int jj = last; jj >= 0 && jj > last - NS; --jj) {
                    drain(bar(B_KFULL + jj % NS), (jj / NS) & 1);
                    drain(bar(B_VFULL + jj % NS), (jj / NS) & 1);
                }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            const uint32_t idesc_s = idesc_bf16(128, KB, 0, 0);   // S, dP: M queries, N keys
            const uint32_t idesc_kv = idesc_bf16(128, 64, 1, 1);  // dV, dK: M keys (A MN-major), N dims (B MN-major)
            const uint32_t idesc_q = idesc_bf16(128, 64, 0, 1);   // dQ: M queries, K keys, N dims (B MN-major)
            // K-major views (K = dims: 32-byte K-steps, +2 in the address field)
            const uint64_t dq_k = sdesc_sw128(sbase + OFF_Q, 16, 1024), ddo_k = sdesc_sw128(sbase + OFF_DO, 16, 1024);
            // MN-major views with K = queries: 16 rows a K-step = 2048 bytes (+128); the
            // 64-key halves of P and dS are TILE bytes apart (the leading byte offset)
            const uint64_t dq_m = sdesc_sw128(sbase + OFF_Q, TILE, 1024), ddo_m = sdesc_sw128(sbase + OFF_DO, TILE, 1024);
            const uint64_t dp_m = sdesc_sw128(sbase + OFF_P, TILE, 1024), dds_m = sdesc_sw128(sbase + OFF_DS, TILE, 1024);
            // dS K-major (K = keys): K-steps 0-3 in the first half, 4-7 in the second
            const uint64_t dds_k = sdesc_sw128(sbase + OFF_DS, 16, 1024);
            bool ok = mbar_wait(bar(B_QFULL), 0, abort_flag, a.status);
            // S = Q K^T and dP = dO V^T of block j (both operands K-major)
            auto issue_sdp = [&](int j) -> bool {
                const int st = j % NS;
                if (!mbar_wait(bar(B_KFULL + st), (j / NS) & 1, abort_flag, a.status) ||
                    !mbar_wait(bar(B_VFULL + st), (j / NS) & 1, abort_flag, a.status))
                    return false;
                tc_fence_after();
                const uint64_t dk_k = sdesc_sw128(sbase + OFF_K + st * TILE, 16, 1024);
                const uint64_t dv_k = sdesc_sw128(sbase + OFF_V + st * TILE, 16, 1024);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) mma_bf16_ss(tmem + T_S, dq_k + 2 * ks, dk_k + 2 * ks, idesc_s, ks > 0);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) mma_bf16_ss(tmem + T_DP, ddo_k + 2 * ks, dv_k + 2 * ks, idesc_s, ks > 0);
                mma_commit(bar(B_SPD));
                return true;
            };
            if (ok && nblk > 0) ok = issue_sdp(0);
            for (int j = 0; ok && j < nblk; ++j) {
                const int st = j % NS;
                // P and dS of block j are in shared memory (S and dP were read before them)
                // and block j - 1's dK, dV are read out
                if (!mbar_wait(bar(B_PDS), j & 1, abort_flag, a.status) ||
                    (j > 0 && !mbar_wait(bar(B_DKVFREE), (j - 1) & 1, abort_flag, a.status))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // the next block's S and dP first: its P and dS are computed while the
                // tensor core runs this block's three products
                if (j + 1 < nblk && !issue_sdp(j + 1)) {
                    ok = false;
                    break;
                }
                const uint64_t dk_m = sdesc_sw128(sbase + OFF_K + st * TILE, TILE, 1024);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) mma_bf16_ss(tmem + T_DV, dp_m + 128 * ks, ddo_m + 128 * ks, idesc_kv, ks > 0);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) mma_bf16_ss(tmem + T_DK, dds_m + 128 * ks, dq_m + 128 * ks, idesc_kv, ks > 0);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks)
                    mma_bf16_ss(tmem + T_DQ, dds_k + (uint64_t)((ks >> 2) * (TILE >> 4) + 2 * (ks & 3)),
                                dk_m + 128 * ks, idesc_q, (j > 0 || ks > 0) ? 1u : 0u);
                mma_commit(bar(B_MMA2));
                mma_commit(bar(B_KVEMPTY + st));
            }
            // every MMA this thread issued completes before the tensor memory is released
            mma_commit(bar(B_FINAL));
            drain(bar(B_FINAL), 0);
        }
    } else {
        // ------------------------------------------------- softmax-gradient rows
        const int wg = (warp - 2) >> 2;     // warpgroup: keys [64 wg, 64 wg + 64), dims [32 wg, 32 wg + 32)
        const int wq = warp & 3;            // tensor-memory lane quarter
        const int rr = wq * 32 + lane;      // query row of the tile; key row of a block
        const uint32_t lb = (uint32_t)(wq * 32) << 16;
        const int64_t p = q0 + rr;
        const bool qv = rr < nq;
        const float sl = a.scale_log2;
        const float L = qv ? a.lse_fwd[row + p] : 0.0f;
        float Dv = 0.0f;  // dout . out of this row
        if (qv) {
            const uint4* o4 = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.out) + (row + p) * D);
            const uint4* g4 = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.dout) + (row + p) * D);
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                const uint4 ow = o4[c8], gw = g4[c8];
                const __nv_bfloat162* ob = reinterpret_cast<const __nv_bfloat162*>(&ow);
                const __nv_bfloat162* gb = reinterpret_cast<const __nv_bfloat162*>(&gw);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float2 of = __bfloat1622float2(ob[u]), gf = __bfloat1622float2(gb[u]);
                    Dv = fmaf(of.x, gf.x, Dv);
                    Dv = fmaf(of.y, gf.y, Dv);
                }
            }
        }
        auto block_keys = [&](int jb, int64_t& t0, int& kv) {
            const bool win = jb >= nbs;
            t0 = win ? ws + (int64_t)KB * (jb - nbs) : (int64_t)KB * jb;
            kv = win ? (int)(q0 + nq - t0 < KB ? q0 + nq - t0 : KB) : (n - KB * jb < KB ? n - KB * jb : KB);
        };
        // dims [32 wg, 32 wg + 32) of the dK and dV rows of block jb to the gradient arrays.
        // The warp's 32 key rows (lane = row in tensor memory) pass through its staging area
        // (16-byte columns XOR-swizzled by row: conflict-free both ways), so that each store
        // or atomic of the warp covers four rows' 128 contiguous bytes instead of one piece
        // of 32 different rows.
        float* stg = reinterpret_cast<float*>(sm + OFF_STG) + (warp - 2) * STG_FLOATS;
        auto spill_rows = [&](const uint32_t (&x)[32], float sc, float* g0, int kv, bool own) {
            __syncwarp();
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
                *reinterpret_cast<float4*>(stg + lane * 32 + ((q4 ^ (lane & 7)) << 2)) =
                    make_float4(__uint_as_float(x[4 * q4]) * sc, __uint_as_float(x[4 * q4 + 1]) * sc,
                                __uint_as_float(x[4 * q4 + 2]) * sc, __uint_as_float(x[4 * q4 + 3]) * sc);
            __syncwarp();
            // step i: rows 4i + r of the warp's 32 (r = lane / 8), 16-byte column c4 = lane % 8;
            // row 4i + r sits at swizzle (4i + r) % 8 = r + 4 (i odd) or r (i even)
            const int c4 = lane & 7, r = lane >> 3, kr0 = wq * 32 + r;
            const float* src0 = stg + r * 32;
            const int col_even = (c4 ^ r) << 2, col_odd = (c4 ^ (r + 4)) << 2;
            float4* dst0 = reinterpret_cast<float4*>(g0 + (int64_t)kr0 * D + 32 * wg) + c4;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 v = *reinterpret_cast<const float4*>(src0 + 128 * i + ((i & 1) ? col_odd : col_even));
                if (kr0 + 4 * i < kv) {
                    float4* dst = dst0 + i * D;  // four rows of D floats = D float4s further
                    if (own)
                        *dst = v;
                    else
                        atomicAdd(dst, v);
                }
            }
        };
        auto readout = [&](int jb) {
            int64_t t0;
            int kv;
            block_keys(jb, t0, kv);
            const bool win = jb >= nbs;
            float* gk = win ? a.dk + (row + t0) * D : a.dks + (((int64_t)bh * a.E + e) * a.M + t0) * D;
            float* gv = win ? a.dv + (row + t0) * D : a.dvs + (((int64_t)bh * a.E + e) * a.M + t0) * D;
            // a read row of the state is this tile's alone when the chunk is one tile
            // (plain stores; the rows were not zeroed); window keys take the sums of
            // every tile that sees them
            const bool own = !win && a.C == TQ;
            uint32_t x[32];
            tmem_ld32(tmem + lb + T_DK + 32 * wg, x);
            tmem_wait_ld();
            spill_rows(x, a.inv_sqrt_d, gk, kv, own);
            tmem_ld32(tmem + lb + T_DV + 32 * wg, x);
            tmem_wait_ld();
            spill_rows(x, 1.0f, gv, kv, own);
        };
        const float2 sl2 = make_float2(sl, sl), nl2 = make_float2(-L, -L);
        bool ok = true;
        for (int j = 0; j < nblk; ++j) {
            int64_t t0;
            int kv;
            block_keys(j, t0, kv);
            // keys [0, lim) of the block are valid for this query (window: causal)
            int lim = 0;
            if (qv) {
                if (j >= nbs) {
                    const int64_t dd = p - t0 + 1;
                    lim = dd < 0 ? 0 : (dd < kv ? (int)dd : kv);
                } else {
                    lim = kv;
                }
            }
            if (!mbar_wait(bar(B_SPD), j & 1, abort_flag, a.status)) { ok = false; break; }
            tc_fence_after();
            // P and dS of keys [64 wg, 64 wg + 64) into registers, 32 keys at a time (the
            // tensor core runs block j - 1's dV, dK, dQ meanwhile)
            uint32_t pw[2][16], dw[2][16];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t sv[32], dp[32];
                tmem_ld32(tmem + lb + T_S + 64 * wg + 32 * h, sv);
                tmem_ld32(tmem + lb + T_DP + 64 * wg + 32 * h, dp);
                tmem_wait_ld();
                const int kb = 64 * wg + 32 * h;
#pragma unroll
                for (int x = 0; x < 32; x += 2) {
                    const float2 t2 = __ffma2_rn(make_float2(__uint_as_float(sv[x]), __uint_as_float(sv[x + 1])), sl2, nl2);
                    const float p0 = kb + x < lim ? ex2(t2.x) : 0.0f;
                    const float p1 = kb + x + 1 < lim ? ex2(t2.y) : 0.0f;
                    const float d0 = p0 * (__uint_as_float(dp[x]) - Dv), d1 = p1 * (__uint_as_float(dp[x + 1]) - Dv);
                    pw[h][x >> 1] = packbf2(p0, p1);
                    dw[h][x >> 1] = packbf2(d0, d1);
                }
            }
            if (j > 0) {
                // block j - 1's products are done: P and dS are free, its dK and dV final
                if (!mbar_wait(bar(B_MMA2), (j - 1) & 1, abort_flag, a.status)) { ok = false; break; }
                tc_fence_after();
                readout(j - 1);
                tc_fence_before();
                mbar_arrive(bar(B_DKVFREE));
            }
            // P and dS of this block into half tile wg (row rr)
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const int chunk = h * 4 + cc;  // 16-byte chunk of the 128-byte half row
                    const uint32_t off = (uint32_t)(wg * TILE + rr * 128 + ((chunk ^ (rr & 7)) << 4));
                    *reinterpret_cast<uint4*>(sm + OFF_P + off) =
                        make_uint4(pw[h][4 * cc], pw[h][4 * cc + 1], pw[h][4 * cc + 2], pw[h][4 * cc + 3]);
                    *reinterpret_cast<uint4*>(sm + OFF_DS + off) =
                        make_uint4(dw[h][4 * cc], dw[h][4 * cc + 1], dw[h][4 * cc + 2], dw[h][4 * cc + 3]);
                }
            // the S and dP loads above complete before the MMA thread may overwrite them
            tc_fence_before();
            fence_proxy_async();  // P and dS (generic-proxy writes) before the MMAs read them
            mbar_arrive(bar(B_PDS));
        }
        if (ok && nblk > 0) {
            if (mbar_wait(bar(B_MMA2), (nblk - 1) & 1, abort_flag, a.status)) {
                tc_fence_after();
                readout(nblk - 1);
                // dims [32 wg, 32 wg + 32) of dq for this row: scaled, rotated back
                // (rotate-half pairs within the row: the whole dQ row is loaded)
                float y[64];
                {
                    uint32_t v0[32], v1[32];
                    tmem_ld32(tmem + lb + T_DQ, v0);
                    tmem_ld32(tmem + lb + T_DQ + 32, v1);
                    tmem_wait_ld();
#pragma unroll
                    for (int x = 0; x < 32; ++x) {
                        y[x] = __uint_as_float(v0[x]) * a.inv_sqrt_d;
                        y[32 + x] = __uint_as_float(v1[x]) * a.inv_sqrt_d;
                    }
                }
                if (qv) {
                    const int half = a.r / 2;
                    float4* dst = reinterpret_cast<float4*>(a.dq + (row + p) * D + 32 * wg);
#pragma unroll
                    for (int x4 = 0; x4 < 8; ++x4) {
                        float o[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int x = 32 * wg + 4 * x4 + u;
                            float v = y[x];
                            if (x < 2 * half) {
                                const int i2 = x < half ? x : x - half;
                                const float2 cs = a.rope[p * half + i2];
                                v = x < half ? y[x] * cs.x + y[x + half] * cs.y : y[x] * cs.x - y[x - half] * cs.y;
                            }
                            o[u] = v;
                        }
                        dst[x4] = make_float4(o[0], o[1], o[2], o[3]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace bwt

// The read rows' gradients need no zeroing when the chunk is exactly one 128-query tile:
// the tile of chunk e + W/C + 1 stores every row of event e below its slot count, the rows
// the slot sweep reads.
bool bwd_tc5_owns_read_rows(const BackwardArgs& a) { return a.C == bwt::TQ; }

bool bwd_tc5_supported(const BackwardArgs& a, bool bf16) {
    return bf16 && a.C % 128 == 0 && a.lse_fwd != nullptr && a.N > 0 && (a.r % 2) == 0;
}

cudaError_t launch_bwd_tc5(const BackwardArgs& a, cudaStream_t s) {
    using namespace bwt;
    CUtensorMap mq, mdo, mk, mv, msk, msv;
    const uint64_t BH = (uint64_t)a.BH, N = (uint64_t)a.N;
    const uint64_t planes_snap = BH * (uint64_t)(a.snap_events > 0 ? a.snap_events : 1);
    if (!make_tmap_bf16_3d(&mq, a.qr, N, BH, TQ) || !make_tmap_bf16_3d(&mdo, a.dout, N, BH, TQ) ||
        !make_tmap_bf16_3d(&mk, a.kr, N, BH, KB) || !make_tmap_bf16_3d(&mv, a.v, N, BH, KB) ||
        !make_tmap_bf16_3d(&msk, a.snap_k, (uint64_t)a.M, planes_snap, KB) ||
        !make_tmap_bf16_3d(&msv, a.snap_v, (uint64_t)a.M, planes_snap, KB))
        return cudaErrorInvalidValue;
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(bwd_tc5_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        attr = true;
    }
    const int tiles = (int)((a.N + TQ - 1) / TQ);
    bwd_tc5_kernel<<<(unsigned)(a.BH * tiles), NTHREADS, SMEM_BYTES, s>>>(mq, mdo, mk, mv, msk, msv, a);
    return cudaGetLastError();
}

}  // namespace kvm
