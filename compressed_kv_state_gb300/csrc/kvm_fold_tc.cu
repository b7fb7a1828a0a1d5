// Fold chain on the tensor cores with the state resident on chip (bf16 I/O,
// chunk <= 128, max_slots <= 256).
//
// "Key-Value Means" (gist.science technical summary), Core mechanisms 1-3
// and 5; lay part "smart merge".  Same rule as the portable fold chain
// (kvm_fold.cu); this kernel keeps one (b, h) row's whole state on one SM
// for the entire chain:
//   - raw fp32 sums in tensor memory: slot j lives in TMEM lane j % 128 of
//     column block j / 128 (64 columns of sum_k, 64 of sum_v); thread j of the
//     CTA owns slot j and is the only one that reads or writes it;
//   - the winner-take-all direction u_j = unit(sum_k_j - mean) in shared
//     memory as two bf16 terms hi + lo (the K-major B operand of the MMA);
//   - the similarity of the 128 chunk keys to all 256 slots is one tcgen05
//     MMA chain S = k (u_hi + u_lo)^T into the other 256 TMEM columns (keys
//     are exactly bf16; the two-term split keeps the cosine to about 1e-6);
//   - the read view (LayerNorm'd keys with the rotary dims zeroed, values at
//     the read radius) in shared memory, recomputed only for slots the event
//     touched, and bulk-copied asynchronously to the event's snapshot;
//   - the next chunk's keys and values arrive by TMA while an event runs.
// The merge is deterministic: each slot's owner thread adds its tokens in
// position order.
#include "kvm_internal.cuh"
#include "tc_primitives.cuh"

namespace kvm {
namespace foldtc {

using namespace tc;

constexpr int MAXS = 256;  // slots held on chip
constexpr int TOK = 128;   // token rows of the MMA tile
constexpr int ROWB = 128;  // bytes of one 64-dim bf16 row
constexpr int OFF_UHI = 0;                      // [256][128 B] swizzled (MMA B operand)
constexpr int OFF_ULO = OFF_UHI + MAXS * ROWB;  // [256][128 B] swizzled
constexpr int OFF_K = OFF_ULO + MAXS * ROWB;    // 2 x [128][128 B] swizzled chunk keys
constexpr int OFF_V = OFF_K + 2 * TOK * ROWB;   // 2 x [128][128 B] swizzled chunk values
constexpr int OFF_VK = OFF_V + 2 * TOK * ROWB;  // [256][128 B] read-view keys (plain rows)
constexpr int OFF_VV = OFF_VK + MAXS * ROWB;    // [256][128 B] read-view values (plain rows)
constexpr int OFF_MISC = OFF_VV + MAXS * ROWB;

struct Misc {
    float g[TOK], kn[TOK], m[TOK];
    float pb[2][TOK], ps[2][TOK];
    int pa[2][TOK];
    int kind[TOK], slot[TOK], list[TOK];
    int hist[4][MAXS];  // merged tokens per slot, per token warp
    int cnt[MAXS];
    float rho[MAXS];
    int cnt_new[MAXS];
    int seg[MAXS + 1];
    int slot_tok[MAXS];
    unsigned long long bar_k[2];
    unsigned long long bar_s;
    uint32_t tmem_slot;
    int abort_flag;
};
constexpr int SMEM_BYTES = OFF_MISC + (int)sizeof(Misc) + 1024;

#ifdef KVM_PROBE
static __device__ unsigned long long g_probe_fold[16];
#endif

__device__ __forceinline__ int swz(int row, int ch) { return row * ROWB + (((ch ^ (row & 7)) & 7) << 4); }

// 64 bf16 of a swizzled row -> fp32
__device__ __forceinline__ void load_row_sw(const uint8_t* base, int row, float (&x)[64]) {
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        const uint4 w = *reinterpret_cast<const uint4*>(base + swz(row, ch));
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float2 f = __bfloat1622float2(h[u]);
            x[ch * 8 + 2 * u] = f.x;
            x[ch * 8 + 2 * u + 1] = f.y;
        }
    }
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Sums over 64 registers with eight independent partial sums (short dependency chains).
__device__ __forceinline__ float sum64(const float (&x)[64]) {
    float p[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) p[i] = x[i];
#pragma unroll
    for (int i = 8; i < 64; ++i) p[i & 7] += x[i];
    return ((p[0] + p[1]) + (p[2] + p[3])) + ((p[4] + p[5]) + (p[6] + p[7]));
}
// sum over x of (x - c)^2, eight partial sums
__device__ __forceinline__ float sqdev64(const float (&x)[64], float c, float scale) {
    float p[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float d = x[i] * scale - c;
        p[i] = d * d;
    }
#pragma unroll
    for (int i = 8; i < 64; ++i) {
        const float d = x[i] * scale - c;
        p[i & 7] = fmaf(d, d, p[i & 7]);
    }
    return ((p[0] + p[1]) + (p[2] + p[3])) + ((p[4] + p[5]) + (p[6] + p[7]));
}
// dot product of two 64-vectors, eight partial sums
__device__ __forceinline__ float dot64(const float (&x)[64], const float (&y)[64]) {
    float p[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) p[i] = x[i] * y[i];
#pragma unroll
    for (int i = 8; i < 64; ++i) p[i & 7] = fmaf(x[i], y[i], p[i & 7]);
    return ((p[0] + p[1]) + (p[2] + p[3])) + ((p[4] + p[5]) + (p[6] + p[7]));
}

// Owner-thread renormalisation of slot j from its key sums (registers): the
// winner-take-all direction u = c / |c| (as bf16 hi + lo terms) and the
// read-view key LayerNorm(sum / count) = c / sqrt(|c|^2 / 64 + eps * count^2),
// both from the centred sums c = sum - mean(sum); rotary dims of the key are 0.
__device__ __forceinline__ void owner_view_k(int j, const float (&sk)[64], int cnt, int r, float eps, uint8_t* sm) {
    const float mean = sum64(sk) * (1.0f / 64.0f);
    float c[64];
#pragma unroll
    for (int x = 0; x < 64; ++x) c[x] = sk[x] - mean;
    const float ss = dot64(c, c);
    const float inv = ss > 0.0f ? 1.0f / sqrtf(ss) : 0.0f;
    const float fc = (float)cnt;
    const float rs = 1.0f / sqrtf(ss * (1.0f / 64.0f) + eps * fc * fc);
    uint4* vk = reinterpret_cast<uint4*>(sm + OFF_VK + j * ROWB);
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        uint32_t hi[4], lo[4], wk[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int x0 = ch * 8 + 2 * u;
            const float a0 = c[x0] * inv, a1 = c[x0 + 1] * inv;
            const __nv_bfloat162 h = __floats2bfloat162_rn(a0, a1);
            const float2 hf = __bfloat1622float2(h);
            const __nv_bfloat162 lw = __floats2bfloat162_rn(a0 - hf.x, a1 - hf.y);
            hi[u] = *reinterpret_cast<const uint32_t*>(&h);
            lo[u] = *reinterpret_cast<const uint32_t*>(&lw);
            wk[u] = (x0 + 1 < r) ? 0u : pack2(x0 < r ? 0.0f : c[x0] * rs, c[x0 + 1] * rs);
        }
        *reinterpret_cast<uint4*>(sm + OFF_UHI + swz(j, ch)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(sm + OFF_ULO + swz(j, ch)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        vk[ch] = make_uint4(wk[0], wk[1], wk[2], wk[3]);
    }
}

// Read-view value of slot j: rho * unit(sum_v).
__device__ __forceinline__ void owner_view_v(int j, const float (&sv)[64], float rho, uint8_t* sm) {
    const float nv = sqrtf(dot64(sv, sv));
    const float f = nv > 0.0f ? rho / nv : 0.0f;
    uint4* vv = reinterpret_cast<uint4*>(sm + OFF_VV + j * ROWB);
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        uint32_t wv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) wv[u] = pack2(sv[ch * 8 + 2 * u] * f, sv[ch * 8 + 2 * u + 1] * f);
        vv[ch] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    }
}

__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&x)[64]) {
    uint32_t a[32], b[32];
    tmem_ld32(taddr, a);
    tmem_ld32(taddr + 32, b);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        x[i] = __uint_as_float(a[i]);
        x[32 + i] = __uint_as_float(b[i]);
    }
}
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const float (&x)[64]) {
    uint32_t a[32], b[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        a[i] = __float_as_uint(x[i]);
        b[i] = __float_as_uint(x[32 + i]);
    }
    tmem_st32(taddr, a);
    tmem_st32(taddr + 32, b);
}

__global__ void __launch_bounds__(256, 1)
    fold_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const FoldArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    Misc& X = *reinterpret_cast<Misc*>(sm + OFF_MISC);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int bh = blockIdx.x;
    const int C = a.C, S = a.S, M = a.M;

    float* g_sum_k = a.sum_k + (int64_t)bh * M * D;
    float* g_sum_v = a.sum_v + (int64_t)bh * M * D;
    int* g_counts = a.counts + (int64_t)bh * M;
    float* g_rho = a.rho + (int64_t)bh * M;
    float* g_simdir = a.simdir + (int64_t)bh * M * D;
    uint8_t* g_view_k = reinterpret_cast<uint8_t*>(a.view_k) + (int64_t)bh * M * ROWB;
    uint8_t* g_view_v = reinterpret_cast<uint8_t*>(a.view_v) + (int64_t)bh * M * ROWB;

    if (tid == 0) {
        mbar_init(smem_u32(&X.bar_k[0]), 1);
        mbar_init(smem_u32(&X.bar_k[1]), 1);
        mbar_init(smem_u32(&X.bar_s), 1);
        X.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(smem_u32(&X.tmem_slot), 512);
    for (int i = tid; i < 2 * MAXS * ROWB / 16; i += 256) {
        reinterpret_cast<uint4*>(sm + OFF_UHI)[i] = make_uint4(0, 0, 0, 0);
        reinterpret_cast<uint4*>(sm + OFF_VK)[i] = make_uint4(0, 0, 0, 0);
    }
    X.cnt[tid] = 0;
    X.rho[tid] = 0.0f;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = X.tmem_slot;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int blk = tid >> 7;  // slot block of the owner thread
    const uint32_t t_sums = tmem + lane_base + blk * 128;
    const uint32_t t_sim = tmem + lane_base + 256;
    const uint32_t sK = smem_u32(sm + OFF_K), sV = smem_u32(sm + OFF_V);
    const uint32_t sUH = smem_u32(sm + OFF_UHI), sUL = smem_u32(sm + OFF_ULO);
    const uint32_t bar_s = smem_u32(&X.bar_s);

    // state before the first event (non-empty for a decode-boundary fold)
    const Sched sc_first = a.sched ? a.sched[a.e_begin] : a.sched0;
    int n = sc_first.n_before;
    {
        const int j = tid;
        float x64[64];
        if (j < n) {
            X.cnt[j] = g_counts[j];
            X.rho[j] = g_rho[j];
        }
#pragma unroll
        for (int x = 0; x < 64; ++x) x64[x] = j < n ? g_sum_k[(int64_t)j * D + x] : 0.0f;
        if (j < n) owner_view_k(j, x64, X.cnt[j], a.r, a.ln_eps, sm);
        tmem_st64(t_sums, x64);
#pragma unroll
        for (int x = 0; x < 64; ++x) x64[x] = j < n ? g_sum_v[(int64_t)j * D + x] : 0.0f;
        if (j < n) owner_view_v(j, x64, X.rho[j], sm);
        tmem_st64(t_sums + 64, x64);
        tmem_wait_st();
    }
    tc_fence_before();
    fence_proxy_async();
    __syncthreads();
    tc_fence_after();

    auto load_chunk = [&](int e, int buf) {
        const int64_t off = ((int64_t)e * C) % a.src_len;
        mbar_expect_tx(smem_u32(&X.bar_k[buf]), 2 * TOK * ROWB);
        tma_load_3d(sK + buf * TOK * ROWB, &tm_k, 0, (int)off, bh, smem_u32(&X.bar_k[buf]));
        tma_load_3d(sV + buf * TOK * ROWB, &tm_v, 0, (int)off, bh, smem_u32(&X.bar_k[buf]));
    };
    if (tid == 0 && a.e_begin < a.e_end && !a.test_stall) load_chunk(a.e_begin, 0);
    const uint32_t idesc = idesc_bf16(128, 256, 0, 0);
    int mma_count = 0;
    KVM_PROBE_DECL(13)
    KVM_PROBE_START()

    // the next event's schedule entry and gates are loaded one event ahead, off the chain
    Sched sc_nx = a.sched ? a.sched[a.e_begin] : a.sched0;
    float g_nx = 0.0f;
    if (tid < C && a.e_begin < a.e_end)
        g_nx = a.g_src[(int64_t)bh * a.src_row + ((int64_t)a.e_begin * C) % a.src_len + tid];
    for (int e = a.e_begin, it = 0; e < a.e_end; ++e, ++it) {
        const int buf = it & 1;
        const Sched sc = sc_nx;
        const float g_here = g_nx;
        if (tid == 0 && !mbar_wait(smem_u32(&X.bar_k[buf]), (it >> 1) & 1, &X.abort_flag, a.status))
            X.abort_flag = 1;
        if (e + 1 < a.e_end) {
            sc_nx = a.sched ? a.sched[e + 1] : a.sched0;
            if (tid < C) g_nx = a.g_src[(int64_t)bh * a.src_row + ((int64_t)(e + 1) * C) % a.src_len + tid];
        }
        __syncthreads();
        if (X.abort_flag) break;
        KVM_PROBE_LAP(0)
#ifdef KVM_PROBE
        probe_acc[8] += 1;
#endif
        const int64_t first_pos = (int64_t)e * C;
        const uint8_t* kch = sm + OFF_K + buf * TOK * ROWB;
        const uint8_t* vch = sm + OFF_V + buf * TOK * ROWB;
        const int n0 = sc.n0, na = sc.a;
        const bool do_mma = n0 > S;

        // similarity of the chunk's keys to every slot direction
        if (do_mma && tid == 0) {
            tc_fence_after();
            for (int ks = 0; ks < 4; ++ks)
                for (int part = 0; part < 2; ++part) {
                    const uint64_t ad = sdesc_sw128(sK + buf * TOK * ROWB + ks * 32, 16, 1024);
                    const uint64_t bd = sdesc_sw128((part ? sUL : sUH) + ks * 32, 16, 1024);
                    mma_bf16_ss(tmem + 256, ad, bd, idesc, (ks | part) ? 1u : 0u);
                }
            mma_commit(bar_s);
        }
        // the next chunk's keys and values load while this event runs
        if (tid == 0 && e + 1 < a.e_end) load_chunk(e + 1, buf ^ 1);
        // per-token set-up
        if (tid < C) {
            const int t = tid;
            X.g[t] = g_here;
            float kx[64];
            load_row_sw(kch, t, kx);
            X.kn[t] = sqrtf(dot64(kx, kx));
            const bool sink = first_pos + t < S;
            X.kind[t] = sink ? 2 : -1;
            X.slot[t] = sink ? (int)(first_pos + t) : -1;
        }
        X.slot_tok[tid] = -1;
#pragma unroll
        for (int w = 0; w < 4; ++w) X.hist[w][tid] = 0;
        __syncthreads();
        KVM_PROBE_LAP(1)

        // best / second / argmax over the mergeable slots [S, n0): each half of
        // the CTA scans 128 slot columns of every token row
        if (do_mma) {
            if (tid == 0 && !mbar_wait(bar_s, mma_count & 1, &X.abort_flag, a.status)) X.abort_flag = 1;
            __syncthreads();
            if (X.abort_flag) break;
            KVM_PROBE_LAP(9)
            ++mma_count;
            tc_fence_after();
            const int half = tid >> 7, t = tid & 127;
            const int lo = max(S, half * 128), hi = min(n0, half * 128 + 128);
            // four independent chains (one per 32-column chunk), merged in index order
            float bq[4], sq[4];
            int aq[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                bq[c] = -INFINITY;
                sq[c] = -INFINITY;
                aq[c] = -1;
            }
            if (lo < hi) {
                uint32_t va[4][32];
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(t_sim + half * 128 + c * 32, va[c]);
                tmem_wait_ld();
                KVM_PROBE_LAP(11)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int base = half * 128 + c * 32;
                    // branchless running best / second best / argmax (strictly larger
                    // values take the lead, so ties keep the lower slot index)
                    if (base >= lo && base + 32 <= hi) {
#pragma unroll
                        for (int x = 0; x < 32; ++x) {
                            const float val = __uint_as_float(va[c][x]);
                            aq[c] = val > bq[c] ? base + x : aq[c];
                            sq[c] = fmaxf(sq[c], fminf(val, bq[c]));
                            bq[c] = fmaxf(bq[c], val);
                        }
                    } else if (base + 32 > lo && base < hi) {
#pragma unroll
                        for (int x = 0; x < 32; ++x) {
                            const int j = base + x;
                            const float val = (j >= lo && j < hi) ? __uint_as_float(va[c][x]) : -INFINITY;
                            aq[c] = val > bq[c] ? j : aq[c];
                            sq[c] = fmaxf(sq[c], fminf(val, bq[c]));
                            bq[c] = fmaxf(bq[c], val);
                        }
                    }
                }
            }
            float b = bq[0], s2 = sq[0];
            int ba = aq[0];
#pragma unroll
            for (int c = 1; c < 4; ++c) {
                if (aq[c] < 0) continue;
                if (ba < 0 || bq[c] > b) {  // a strictly larger value from a later chunk wins
                    s2 = fmaxf(fmaxf(s2, sq[c]), ba < 0 ? -INFINITY : b);
                    b = bq[c];
                    ba = aq[c];
                } else {
                    s2 = fmaxf(s2, bq[c]);
                    s2 = fmaxf(s2, sq[c]);
                }
            }
            KVM_PROBE_LAP(12)
            X.pb[half][t] = b;
            X.ps[half][t] = s2;
            X.pa[half][t] = ba;
            tc_fence_before();
            __syncthreads();
        }
        KVM_PROBE_LAP(2)
        float best = -INFINITY, sec = -INFINITY;
        int barg = -1;
        const bool cand = tid < C && X.kind[tid] != 2;
        if (cand && do_mma) {
            const int t = tid;
            const float b0 = X.pb[0][t], s0 = X.ps[0][t], b1 = X.pb[1][t], s1 = X.ps[1][t];
            const int a0 = X.pa[0][t], a1 = X.pa[1][t];
            if (a0 >= 0 && (a1 < 0 || b0 >= b1)) {
                best = b0;
                barg = a0;
                sec = fmaxf(s0, a1 >= 0 ? b1 : -INFINITY);
                sec = fmaxf(sec, s1);
            } else if (a1 >= 0) {
                best = b1;
                barg = a1;
                sec = fmaxf(s1, a0 >= 0 ? b0 : -INFINITY);
                sec = fmaxf(sec, s0);
            }
        }
        const float kn = tid < C ? X.kn[tid] : 0.0f;
        if (cand) X.m[tid] = barg < 0 ? -INFINITY : (kn > 0.0f ? best / kn : 0.0f);
        __syncthreads();

        // surprise selection: the a lowest scores (ties to the lower position) are appended
        if (na > 0) {
            int rank = 0;
            if (cand) {
                const float mt = X.m[tid];
#pragma unroll 4
                for (int u = 0; u < C; ++u) {
                    if (X.kind[u] == 2) continue;
                    const float mu = X.m[u];
                    rank += (mu < mt) || (mu == mt && u < tid);
                }
            }
            __syncthreads();
            if (cand) X.kind[tid] = rank < na ? 1 : 0;
            __syncthreads();
            if (tid < C && X.kind[tid] == 1) {
                int before = 0;
                for (int u = 0; u < tid; ++u) before += (X.kind[u] == 1);
                X.slot[tid] = n0 + before;
            }
        } else if (cand) {
            X.kind[tid] = 0;
        }
        __syncthreads();
        if (tid < C && X.kind[tid] != 0) X.slot_tok[X.slot[tid]] = tid;
        __syncthreads();
        KVM_PROBE_LAP(3)

        if (na > 0) {
            // directions of the new slots (from their founding token), then the
            // remaining tokens also compare against them
            const int j = tid;
            if (j >= n0 && j < n0 + na) {
                const int t = X.slot_tok[j];
                float kx[64];
                load_row_sw(kch, t, kx);
                const float g = X.g[t];
#pragma unroll
                for (int x = 0; x < 64; ++x) kx[x] = g * kx[x];
                const float mean = sum64(kx) * (1.0f / 64.0f);
                const float ss = sqdev64(kx, mean, 1.0f);
                const float inv = ss > 0.0f ? 1.0f / sqrtf(ss) : 0.0f;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    uint32_t hw[4], lw[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float a0 = (kx[ch * 8 + 2 * u] - mean) * inv;
                        const float a1 = (kx[ch * 8 + 2 * u + 1] - mean) * inv;
                        const __nv_bfloat16 h0 = __float2bfloat16_rn(a0), h1 = __float2bfloat16_rn(a1);
                        hw[u] = pack2(__bfloat162float(h0), __bfloat162float(h1));
                        lw[u] = pack2(a0 - __bfloat162float(h0), a1 - __bfloat162float(h1));
                    }
                    *reinterpret_cast<uint4*>(sm + OFF_UHI + swz(j, ch)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    *reinterpret_cast<uint4*>(sm + OFF_ULO + swz(j, ch)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                }
            }
            __syncthreads();
            if (tid < C && X.kind[tid] == 0) {
                float kx[64];
                load_row_sw(kch, tid, kx);
                for (int jj = n0; jj < n0 + na; ++jj) {
                    float hx[64], lx[64];
                    load_row_sw(sm + OFF_UHI, jj, hx);
                    load_row_sw(sm + OFF_ULO, jj, lx);
#pragma unroll
                    for (int x = 0; x < 64; ++x) hx[x] += lx[x];
                    const float s = dot64(kx, hx);
                    if (s > best) {
                        sec = best;
                        best = s;
                        barg = jj;
                    } else if (s > sec) {
                        sec = s;
                    }
                }
            }
        }
        if (tid < C && X.kind[tid] == 0) {
            X.slot[tid] = barg;
            if (barg < 0 && a.status) atomicOr(a.status, STATUS_DEVICE);
        }
        if (tid < C && e < a.dbg_events) {
            const int64_t o = ((int64_t)bh * a.dbg_events + e) * C + tid;
            const int kd = X.kind[tid];
            if (a.dbg_assign) a.dbg_assign[o] = X.slot[tid];
            if (a.dbg_kind) a.dbg_kind[o] = kd;
            if (a.dbg_m) a.dbg_m[o] = kd == 2 ? __int_as_float(0x7fc00000) : X.m[tid];
            if (a.dbg_gap) {
                float gp = __int_as_float(0x7fc00000);
                if (kd == 0) gp = sec == -INFINITY ? INFINITY : (kn > 0.0f ? (best - sec) / kn : 0.0f);
                a.dbg_gap[o] = gp;
            }
        }
        __syncthreads();

        KVM_PROBE_LAP(4)
        // merge lists: merged tokens grouped by slot, position order inside a slot.
        // A token's rank among earlier tokens of its slot = earlier lanes of its
        // warp with the same slot (match_any) + the same slot's count in earlier warps.
        int rank_in_slot = 0, sj = -1;
        const bool merged = tid < C && X.kind[tid] == 0 && X.slot[tid] >= 0;
        if (warp < 4) {
            sj = merged ? X.slot[tid] : -1;
            const unsigned same = __match_any_sync(0xffffffffu, merged ? sj : MAXS + (tid & 31));
            const int lane = tid & 31;
            rank_in_slot = __popc(same & ((1u << lane) - 1u));
            if (merged && rank_in_slot == 0) X.hist[warp][sj] = __popc(same);
        }
        __syncthreads();
        if (merged)
            for (int w = 0; w < warp; ++w) rank_in_slot += X.hist[w][sj];
        X.cnt_new[tid] = X.hist[0][tid] + X.hist[1][tid] + X.hist[2][tid] + X.hist[3][tid];
        __syncthreads();
        if (warp == 0) {
            const int lane = tid & 31;
            int v8[8], sacc = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                v8[i] = X.cnt_new[lane * 8 + i];
                sacc += v8[i];
            }
            int incl = sacc;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            int run = incl - sacc;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                X.seg[lane * 8 + i] = run;
                run += v8[i];
            }
            if (lane == 31) X.seg[MAXS] = run;
            // the previous snapshot store must have finished reading the view
            if (lane == 0) bulk_wait_read();
        }
        __syncthreads();
        if (merged) X.list[X.seg[sj] + rank_in_slot] = tid;
        __syncthreads();
        KVM_PROBE_LAP(5)

        // owner threads: founding and merging into their slot, then the new read view
        {
            const int j = tid;
            const int ft = X.slot_tok[j];
            const int nm = X.cnt_new[j];
            const bool touched = ft >= 0 || nm > 0;
            if (__any_sync(0xffffffffu, touched)) {
                const int b0 = X.seg[j];
                int cnt = X.cnt[j];
                float rho = X.rho[j];
                float x64[64], tx[64];
                // keys
                tmem_ld64(t_sums, x64);
                if (touched) {
                    if (ft >= 0) {
                        load_row_sw(kch, ft, tx);
                        const float g = X.g[ft];
#pragma unroll
                        for (int x = 0; x < 64; ++x) x64[x] = g * tx[x];
                        cnt = 0;
                    }
                    // merged tokens in position order
                    for (int i = b0; i < b0 + nm; ++i) {
                        const int t = X.list[i];
                        load_row_sw(kch, t, tx);
                        const float g = X.g[t];
#pragma unroll
                        for (int x = 0; x < 64; ++x) x64[x] = fmaf(g, tx[x], x64[x]);
                    }
                    cnt += nm + (ft >= 0 ? 1 : 0);
                    owner_view_k(j, x64, cnt, a.r, a.ln_eps, sm);
                }
                tmem_st64(t_sums, x64);
                // values
                tmem_ld64(t_sums + 64, x64);
                if (touched) {
                    if (ft >= 0) {
                        load_row_sw(vch, ft, tx);
                        const float g = X.g[ft];
#pragma unroll
                        for (int x = 0; x < 64; ++x) x64[x] = g * tx[x];
                        rho = sqrtf(dot64(tx, tx));
                    }
                    for (int i = b0; i < b0 + nm; ++i) {
                        const int t = X.list[i];
                        load_row_sw(vch, t, tx);
                        const float g = X.g[t];
#pragma unroll
                        for (int x = 0; x < 64; ++x) x64[x] = fmaf(g, tx[x], x64[x]);
                    }
                    owner_view_v(j, x64, rho, sm);
                    X.cnt[j] = cnt;
                    X.rho[j] = rho;
                }
                tmem_st64(t_sums + 64, x64);
                tmem_wait_st();
            }
        }
        KVM_PROBE_LAP(6)
        tc_fence_before();
        fence_proxy_async();
        __syncthreads();
        tc_fence_after();

        // snapshot of the read view after this event (async bulk copy)
        if (tid == 0 && a.snap_k && e < a.snap_events) {
            const int64_t base = ((int64_t)bh * a.snap_events + e) * M * ROWB;
            const uint32_t bytes = (uint32_t)sc.n_after * ROWB;
            bulk_store(reinterpret_cast<uint8_t*>(a.snap_k) + base, smem_u32(sm + OFF_VK), bytes);
            bulk_store(reinterpret_cast<uint8_t*>(a.snap_v) + base, smem_u32(sm + OFF_VV), bytes);
            bulk_commit();
        }
        n = sc.n_after;
        KVM_PROBE_LAP(7)
    }

    // write the state back for decode, export and the portable kernels
    if (tid == 0) bulk_wait_all();
    {
        const int j = tid;
        const bool wr = j < n && !X.abort_flag;
        float x64[64];
        tmem_ld64(t_sums, x64);
        if (wr) {
            const float mean = sum64(x64) * (1.0f / 64.0f);
            const float ss = sqdev64(x64, mean, 1.0f);
            const float inv = ss > 0.0f ? 1.0f / sqrtf(ss) : 0.0f;
            float4* dk = reinterpret_cast<float4*>(g_sum_k + (int64_t)j * D);
            float4* ds = reinterpret_cast<float4*>(g_simdir + (int64_t)j * D);
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                dk[x] = make_float4(x64[4 * x], x64[4 * x + 1], x64[4 * x + 2], x64[4 * x + 3]);
                ds[x] = make_float4((x64[4 * x] - mean) * inv, (x64[4 * x + 1] - mean) * inv,
                                    (x64[4 * x + 2] - mean) * inv, (x64[4 * x + 3] - mean) * inv);
            }
        }
        tmem_ld64(t_sums + 64, x64);
        if (wr) {
            float4* dv = reinterpret_cast<float4*>(g_sum_v + (int64_t)j * D);
#pragma unroll
            for (int x = 0; x < 16; ++x) dv[x] = make_float4(x64[4 * x], x64[4 * x + 1], x64[4 * x + 2], x64[4 * x + 3]);
            g_counts[j] = X.cnt[j];
            g_rho[j] = X.rho[j];
            const uint4* vk = reinterpret_cast<const uint4*>(sm + OFF_VK + j * ROWB);
            const uint4* vv = reinterpret_cast<const uint4*>(sm + OFF_VV + j * ROWB);
            uint4* gk = reinterpret_cast<uint4*>(g_view_k + (int64_t)j * ROWB);
            uint4* gv = reinterpret_cast<uint4*>(g_view_v + (int64_t)j * ROWB);
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                gk[ch] = vk[ch];
                gv[ch] = vv[ch];
            }
        }
    }
    KVM_PROBE_LAP(10)
    if (tid == 0) KVM_PROBE_FLUSH(g_probe_fold, 0, 13)
    tc_fence_before();
    __syncthreads();
    if (X.abort_flag) {
        const long long t0 = clock64();
        while (clock64() - t0 < (1ll << 22)) {
        }
    }
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace foldtc

KVM_PROBE_READOUT(kvm_probe_read_fold, foldtc::g_probe_fold)

bool fold_tc_supported(const FoldArgs& a, bool bf16) { return bf16 && a.C <= 128 && a.M <= foldtc::MAXS; }

cudaError_t launch_fold_tc(const FoldArgs& a, cudaStream_t s) {
    CUtensorMap mk, mv;
    if (!make_tmap_bf16_3d(&mk, a.k_src, (uint64_t)a.src_row, (uint64_t)a.BH, 128) ||
        !make_tmap_bf16_3d(&mv, a.v_src, (uint64_t)a.src_row, (uint64_t)a.BH, 128))
        return cudaErrorInvalidValue;
    cudaFuncSetAttribute(foldtc::fold_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, foldtc::SMEM_BYTES);
    foldtc::fold_tc_kernel<<<a.BH, 256, foldtc::SMEM_BYTES, s>>>(mk, mv, a);
    return cudaGetLastError();
}

}  // namespace kvm
