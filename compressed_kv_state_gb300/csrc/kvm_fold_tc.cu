// Fold chain on the tensor cores with the state resident on chip (bf16 I/O,
// chunk <= 128, max_slots <= 256).
//
// "Key-Value Means" (gist.science technical summary), Core mechanisms 1-3
// and 5; lay part "smart merge".  Same rule as the portable fold chain
// (kvm_fold.cu); this kernel keeps one (b, h) row's whole state on one SM
// for the entire chain, with 512 threads:
//   - raw fp32 sums in tensor memory: slot j lives in TMEM lane j % 128 of
//     column block j / 128 (64 columns of sum_k, 64 of sum_v); thread j owns
//     the key sums of slot j and thread 256 + j its value sums (the same TMEM
//     lane: warps w and w + 8 address the same lane quarter), and nobody else
//     reads or writes them;
//   - the winner-take-all direction u_j = unit(sum_k_j - mean) in shared
//     memory as two bf16 terms hi + lo (the K-major B operand of the MMA);
//   - the similarity of the 128 chunk keys to all 256 slots is one tcgen05
//     MMA chain S = k (u_hi + u_lo)^T into the other 256 TMEM columns (keys
//     are exactly bf16; the two-term split keeps the cosine to about 1e-6);
//     four threads scan each token's row (64 slot columns each);
//   - the read view (LayerNorm'd keys with the rotary dims zeroed, values at
//     the read radius) in shared memory, recomputed only for slots the event
//     touched, and bulk-copied asynchronously to the event's snapshot;
//   - the next chunk's keys and values arrive by TMA while an event runs.
// The merge is deterministic: each slot's owner threads add its tokens in
// position order.  Rows are accumulated 8 dims at a time from shared memory
// so that every thread stays within 128 registers.
#include "kvm_internal.cuh"
#include "tc_primitives.cuh"

namespace kvm {
namespace foldtc {

using namespace tc;

constexpr int MAXS = 256;  // slots held on chip
constexpr int TOK = 128;   // token rows of the MMA tile
constexpr int NT = 512;    // threads: key owner j and value owner 256 + j of every slot j
constexpr int TMA_T = NT - 1;  // issues the chunk loads and the view stores (a value-side
                               // thread: its warp has slack, thread 0 is on the chain)
// A value warp, idle once its own slots are done, issues the next event's similarity MMA
// after the key side's barrier (lane 0), and skips the event's closing barrier: issuing
// holds the thread while the tensor core takes the MMAs, off every other thread's path.
constexpr int MMA_W = 14;
constexpr int ROWB = 128;  // bytes of one 64-dim bf16 row
constexpr int OFF_UHI = 0;                      // [256][128 B] swizzled (MMA B operand)
constexpr int OFF_ULO = OFF_UHI + MAXS * ROWB;  // [256][128 B] swizzled
constexpr int OFF_K = OFF_ULO + MAXS * ROWB;    // 2 x [128][128 B] swizzled chunk keys
constexpr int OFF_V = OFF_K + 2 * TOK * ROWB;   // 2 x [128][128 B] swizzled chunk values
constexpr int OFF_VK = OFF_V + 2 * TOK * ROWB;  // [256][128 B] swizzled read-view keys
constexpr int OFF_VV = OFF_VK + MAXS * ROWB;    // [256][128 B] swizzled read-view values
constexpr int OFF_MISC = OFF_VV + MAXS * ROWB;

struct Misc {
    float g[TOK], kn[TOK], m[TOK];
    float pb[4][TOK], ps[4][TOK];  // best / second best of each 64-slot quarter
    int pa[4][TOK];                // argmax of each quarter
    int kind[TOK], slot[TOK];
    uint32_t tmask[MAXS][4];  // merged tokens of each slot: bit t of the 128-bit mask = token t
    int cnt[MAXS];      // written by key owners
    float rho[MAXS];    // written by value owners
    int cntv[MAXS];     // value owners' copy of the counts (read value of the no-norm ablation)
    int slot_tok[MAXS];
    unsigned long long bar_k[2];
    unsigned long long bar_s;
    unsigned long long bar_st;  // state rows staged by TMA
    uint32_t tmem_slot;
    int abort_flag;
};
constexpr int SMEM_BYTES = OFF_MISC + (int)sizeof(Misc) + 1024;

#ifdef KVM_PROBE
// per-phase cycles of four sample threads (0, 255, 256, 511), 20 counters each
static __device__ unsigned long long g_probe_fold[80];
#endif

__device__ __forceinline__ int swz(int row, int ch) { return row * ROWB + (((ch ^ (row & 7)) & 7) << 4); }

// fp32 state rows move between global memory and shared memory by TMA through
// staging tiles: half h (floats [32h, 32h + 32)) of row j at
// h * 32 KB + j * 128 B, 16-byte chunk c at (c ^ (j & 7)) * 16 (the 128-byte
// swizzle, so that the row-per-thread accesses below are conflict-free).
constexpr int STAGE_ROWS = 64;  // rows per TMA box (fewer when max_slots is smaller)
__device__ __forceinline__ uint32_t stage_off(int j, int q) {
    const int h = q >> 3, c = q & 7;
    return (uint32_t)(h * 32768 + j * 128 + ((c ^ (j & 7)) << 4));
}

__device__ __forceinline__ float2 bf2(uint32_t w) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
}

// x = g * row, for the 64 bf16 of a swizzled row
__device__ __forceinline__ void set_row_sw(const uint8_t* base, int row, float g, float (&x)[64]) {
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        const uint4 w = *reinterpret_cast<const uint4*>(base + swz(row, ch));
        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float2 f = bf2(wv[u]);
            x[ch * 8 + 2 * u] = g * f.x;
            x[ch * 8 + 2 * u + 1] = g * f.y;
        }
    }
}
// x += g * row
__device__ __forceinline__ void add_row_sw(const uint8_t* base, int row, float g, float (&x)[64]) {
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        const uint4 w = *reinterpret_cast<const uint4*>(base + swz(row, ch));
        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float2 f = bf2(wv[u]);
            x[ch * 8 + 2 * u] = fmaf(g, f.x, x[ch * 8 + 2 * u]);
            x[ch * 8 + 2 * u + 1] = fmaf(g, f.y, x[ch * 8 + 2 * u + 1]);
        }
    }
}
// sum of squares of the dims [8 c0, 8 (c0 + nc)) of a swizzled row, partial
// sums by dim mod 8 in increasing dim order (the order of dot64 below)
template <int NC>
__device__ __forceinline__ float sq_row_sw(const uint8_t* base, int row, int c0) {
    float p[8];
#pragma unroll
    for (int ch = 0; ch < NC; ++ch) {
        const uint4 w = *reinterpret_cast<const uint4*>(base + swz(row, c0 + ch));
        const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float2 f = bf2(wv[u]);
            if (ch == 0) {
                p[2 * u] = f.x * f.x;
                p[2 * u + 1] = f.y * f.y;
            } else {
                p[2 * u] = fmaf(f.x, f.x, p[2 * u]);
                p[2 * u + 1] = fmaf(f.y, f.y, p[2 * u + 1]);
            }
        }
    }
    return ((p[0] + p[1]) + (p[2] + p[3])) + ((p[4] + p[5]) + (p[6] + p[7]));
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
// dot product of two 64-vectors, eight partial sums
__device__ __forceinline__ float dot64(const float (&x)[64], const float (&y)[64]) {
    float p[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) p[i] = x[i] * y[i];
#pragma unroll
    for (int i = 8; i < 64; ++i) p[i & 7] = fmaf(x[i], y[i], p[i & 7]);
    return ((p[0] + p[1]) + (p[2] + p[3])) + ((p[4] + p[5]) + (p[6] + p[7]));
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

// ---- packed fp32 (two lanes per instruction, sm_100 family) versions of the
// owner-phase arithmetic.  Pair i holds dims (2i, 2i + 1); every reduction keeps
// the order of the scalar helpers above (partial sums by dim mod 8, combined
// pairwise), and a packed fused multiply-add rounds each lane once exactly like
// fmaf, so the results are the scalar ones bit for bit.
__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 bf2u(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
// x = g * row
__device__ __forceinline__ void set_row_sw2(const uint8_t* base, int row, float g, float2 (&x)[32]) {
    const float2 g2 = f2(g);
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        const uint4 w = *reinterpret_cast<const uint4*>(base + swz(row, ch));
        x[4 * ch + 0] = __fmul2_rn(g2, bf2u(w.x));
        x[4 * ch + 1] = __fmul2_rn(g2, bf2u(w.y));
        x[4 * ch + 2] = __fmul2_rn(g2, bf2u(w.z));
        x[4 * ch + 3] = __fmul2_rn(g2, bf2u(w.w));
    }
}
// x += g * row
__device__ __forceinline__ void add_row_sw2(const uint8_t* base, int row, float g, float2 (&x)[32]) {
    const float2 g2 = f2(g);
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        const uint4 w = *reinterpret_cast<const uint4*>(base + swz(row, ch));
        x[4 * ch + 0] = __ffma2_rn(g2, bf2u(w.x), x[4 * ch + 0]);
        x[4 * ch + 1] = __ffma2_rn(g2, bf2u(w.y), x[4 * ch + 1]);
        x[4 * ch + 2] = __ffma2_rn(g2, bf2u(w.z), x[4 * ch + 2]);
        x[4 * ch + 3] = __ffma2_rn(g2, bf2u(w.w), x[4 * ch + 3]);
    }
}
__device__ __forceinline__ float fold8(const float2 (&p)[4]) {
    return ((p[0].x + p[0].y) + (p[1].x + p[1].y)) + ((p[2].x + p[2].y) + (p[3].x + p[3].y));
}
__device__ __forceinline__ float sum64_2(const float2 (&x)[32]) {
    float2 p[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
    for (int i = 4; i < 32; ++i) p[i & 3] = __fadd2_rn(p[i & 3], x[i]);
    return fold8(p);
}
__device__ __forceinline__ float dot64_2(const float2 (&x)[32], const float2 (&y)[32]) {
    float2 p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = __fmul2_rn(x[i], y[i]);
#pragma unroll
    for (int i = 4; i < 32; ++i) p[i & 3] = __ffma2_rn(x[i], y[i], p[i & 3]);
    return fold8(p);
}
__device__ __forceinline__ uint32_t pack2f(float2 v) { return pack2(v.x, v.y); }

// Key owner, part 1 (on the chain's critical path): centre the key sums in place
// and write the winner-take-all direction u = c / |c| as bf16 hi + lo terms.
// Returns |c|^2.
__device__ __forceinline__ float key_dir2(int j, float2 (&c)[32], uint8_t* sm) {
    const float2 m2 = f2(-(sum64_2(c) * (1.0f / 64.0f)));
#pragma unroll
    for (int i = 0; i < 32; ++i) c[i] = __fadd2_rn(c[i], m2);
    const float ss = dot64_2(c, c);
    const float2 inv = f2(ss > 0.0f ? 1.0f / sqrtf(ss) : 0.0f);
    const float2 neg1 = f2(-1.0f);
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float2 a = __fmul2_rn(c[4 * ch + u], inv);
            hi[u] = pack2f(a);
            lo[u] = pack2f(__ffma2_rn(bf2u(hi[u]), neg1, a));  // a - hi, exact
        }
        *reinterpret_cast<uint4*>(sm + OFF_UHI + swz(j, ch)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(sm + OFF_ULO + swz(j, ch)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    return ss;
}
// Key owner, part 2: the read-view key LayerNorm(sum / count) =
// c / sqrt(|c|^2 / 64 + eps * count^2) with the rotary dims [0, r) zeroed.
__device__ __forceinline__ void key_view2(int j, const float2 (&c)[32], float ss, int cnt, int r, float eps,
                                          uint8_t* sm) {
    const float fc = (float)cnt;
    const float2 rs = f2(1.0f / sqrtf(ss * (1.0f / 64.0f) + eps * fc * fc));
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
        uint32_t wk[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int x0 = ch * 8 + 2 * u;
            const float2 y = __fmul2_rn(c[4 * ch + u], rs);
            wk[u] = (x0 + 1 < r) ? 0u : pack2(x0 < r ? 0.0f : y.x, y.y);
        }
        *reinterpret_cast<uint4*>(sm + OFF_VK + swz(j, ch)) = make_uint4(wk[0], wk[1], wk[2], wk[3]);
    }
}
// Value owner's read view: rho * unit(sum_v) (with the no-norm ablation, the
// member mean sum_v / count: rho < 0 carries -1 / count).
__device__ __forceinline__ void value_view2(int j, const float2 (&sv)[32], float rho, uint8_t* sm) {
    const float nv = sqrtf(dot64_2(sv, sv));
    const float2 f = f2(rho < 0.0f ? -rho : (nv > 0.0f ? rho / nv : 0.0f));
#pragma unroll
    for (int ch = 0; ch < 8; ++ch)
        *reinterpret_cast<uint4*>(sm + OFF_VV + swz(j, ch)) =
            make_uint4(pack2f(__fmul2_rn(sv[4 * ch], f)), pack2f(__fmul2_rn(sv[4 * ch + 1], f)),
                       pack2f(__fmul2_rn(sv[4 * ch + 2], f)), pack2f(__fmul2_rn(sv[4 * ch + 3], f)));
}
__device__ __forceinline__ void tmem_ld64_2(uint32_t taddr, float2 (&x)[32]) {
    uint32_t a[32], b[32];
    tmem_ld32(taddr, a);
    tmem_ld32(taddr + 32, b);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        x[i] = make_float2(__uint_as_float(a[2 * i]), __uint_as_float(a[2 * i + 1]));
        x[16 + i] = make_float2(__uint_as_float(b[2 * i]), __uint_as_float(b[2 * i + 1]));
    }
}
__device__ __forceinline__ void tmem_st64_2(uint32_t taddr, const float2 (&x)[32]) {
    uint32_t a[32], b[32];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        a[2 * i] = __float_as_uint(x[i].x);
        a[2 * i + 1] = __float_as_uint(x[i].y);
        b[2 * i] = __float_as_uint(x[16 + i].x);
        b[2 * i + 1] = __float_as_uint(x[16 + i].y);
    }
    tmem_st32(taddr, a);
    tmem_st32(taddr + 32, b);
}

// Running best / argmax (and, with GAP, second best) over 32 slot columns
// starting at slot base, restricted to [lo, hi); strictly larger values take
// the lead, so ties keep the lower slot index.  The second best only feeds the
// debug record's top-2 gap.
template <bool GAP>
__device__ __forceinline__ void scan32(const uint32_t (&v)[32], int base, int lo, int hi, float& b, float& s,
                                       int& arg) {
    if (base >= lo && base + 32 <= hi) {
#pragma unroll
        for (int x = 0; x < 32; ++x) {
            const float val = __uint_as_float(v[x]);
            arg = val > b ? base + x : arg;
            if (GAP) s = fmaxf(s, fminf(val, b));
            b = fmaxf(b, val);
        }
    } else if (base + 32 > lo && base < hi) {
#pragma unroll
        for (int x = 0; x < 32; ++x) {
            const int j = base + x;
            const float val = (j >= lo && j < hi) ? __uint_as_float(v[x]) : -INFINITY;
            arg = val > b ? j : arg;
            if (GAP) s = fmaxf(s, fminf(val, b));
            b = fmaxf(b, val);
        }
    }
}

// (b, s, arg) <- combination with a later (higher slot index) partial result.
__device__ __forceinline__ void merge_later(float& b, float& s, int& arg, float b2, float s2, int a2) {
    if (a2 < 0) return;
    if (arg < 0 || b2 > b) {
        s = fmaxf(fmaxf(s, s2), arg < 0 ? -INFINITY : b);
        b = b2;
        arg = a2;
    } else {
        s = fmaxf(s, b2);
        s = fmaxf(s, s2);
    }
}

template <bool GAP>
__global__ void __launch_bounds__(NT, 1)
    fold_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const __grid_constant__ CUtensorMap tm_sk, const __grid_constant__ CUtensorMap tm_sv,
                   const __grid_constant__ CUtensorMap tm_snk, const __grid_constant__ CUtensorMap tm_snv,
                   const __grid_constant__ CUtensorMap tm_vv, const FoldArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    Misc& X = *reinterpret_cast<Misc*>(sm + OFF_MISC);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int j = tid & (MAXS - 1);  // owned slot
    const bool vside = tid >= MAXS;  // value owner (else key owner)
    const int bh = blockIdx.x;
    const int C = a.C, S = a.S, M = a.M;

    int* g_counts = a.counts + (int64_t)bh * M;
    float* g_rho = a.rho + (int64_t)bh * M;

    // state before the first event (non-empty for a decode-boundary fold or a later segment)
    const Sched sc_first = a.sched ? a.sched[a.e_begin] : a.sched0;
    int n = sc_first.n_before;
    const int srows = a.stage_rows;
    const int nblk_st = (n + srows - 1) / srows;
    if (tid == 0) {
        mbar_init(smem_u32(&X.bar_k[0]), 1);
        mbar_init(smem_u32(&X.bar_k[1]), 1);
        mbar_init(smem_u32(&X.bar_s), 1);
        mbar_init(smem_u32(&X.bar_st), 1);
        X.abort_flag = 0;
        fence_barrier_init();
        // key sums staged in the direction area, value sums in the read-view area
        if (nblk_st > 0) {
            const uint32_t bst = smem_u32(&X.bar_st);
            mbar_expect_tx(bst, 2 * 2 * nblk_st * srows * 128);
            for (int h = 0; h < 2; ++h)
                for (int b = 0; b < nblk_st; ++b) {
                    const uint32_t o = h * 32768 + b * srows * 128;
                    tma_load_3d(smem_u32(sm + OFF_UHI) + o, &tm_sk, 32 * h, b * srows, bh, bst);
                    tma_load_3d(smem_u32(sm + OFF_VK) + o, &tm_sv, 32 * h, b * srows, bh, bst);
                }
        }
    }
    if (warp == 0) tmem_alloc(smem_u32(&X.tmem_slot), 512);
    if (!vside) {
        X.cnt[j] = 0;
        X.rho[j] = 0.0f;
        X.cntv[j] = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = X.tmem_slot;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    // this thread's sums: slot block j / 128, key columns [0, 64) or value columns [64, 128)
    const uint32_t t_own = tmem + lane_base + (j >> 7) * 128 + (vside ? 64 : 0);
    const uint32_t t_sim = tmem + lane_base + 256;
    const uint32_t sK = smem_u32(sm + OFF_K), sV = smem_u32(sm + OFF_V);
    const uint32_t sUH = smem_u32(sm + OFF_UHI), sUL = smem_u32(sm + OFF_ULO);
    const uint32_t bar_s = smem_u32(&X.bar_s);
    // thread 0's record of asynchronous work it issued that no wait has seen
    // complete yet (phase parity, or -1): drained before the CTA releases its
    // tensor memory after an abort
    int pend_st = -1, pend_ld[2] = {-1, -1}, pend_mma = -1;

    auto load_chunk = [&](int e, int buf) {
        pend_ld[buf] = ((e - a.e_begin) >> 1) & 1;
        const int64_t off = ((int64_t)e * C) % a.src_len;
        mbar_expect_tx(smem_u32(&X.bar_k[buf]), 2 * TOK * ROWB);
        tma_load_3d(sK + buf * TOK * ROWB, &tm_k, 0, (int)off, bh, smem_u32(&X.bar_k[buf]));
        tma_load_3d(sV + buf * TOK * ROWB, &tm_v, 0, (int)off, bh, smem_u32(&X.bar_k[buf]));
    };
    // the first two chunks load now, while the state is restored (the chunk buffers are
    // not staging areas); chunk e + 2 is issued at the end of event e
    if (tid == TMA_T && a.e_begin < a.e_end && !a.test_stall) {
        load_chunk(a.e_begin, 0);
        if (a.e_begin + 1 < a.e_end) load_chunk(a.e_begin + 1, 1);
    }

    {
        float2 x[32];
        if (nblk_st > 0) {
            if (tid == 0 && !mbar_wait(smem_u32(&X.bar_st), 0, &X.abort_flag, a.status)) {
                X.abort_flag = 1;
                pend_st = 0;
            }
            __syncthreads();
        }
        const uint8_t* stage = sm + (vside ? OFF_VK : OFF_UHI);
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const float4 f = (j < n && !X.abort_flag) ? *reinterpret_cast<const float4*>(stage + stage_off(j, q))
                                                      : make_float4(0.f, 0.f, 0.f, 0.f);
            x[2 * q] = make_float2(f.x, f.y);
            x[2 * q + 1] = make_float2(f.z, f.w);
        }
        __syncthreads();  // the staging areas are free again
        tmem_st64_2(t_own, x);
        tmem_wait_st();
        if (j < n) {
            if (!vside) {
                const int cnt = g_counts[j];
                X.cnt[j] = cnt;
                const float ss = key_dir2(j, x, sm);
                key_view2(j, x, ss, cnt, a.r, a.ln_eps, sm);
            } else {
                const float rho = g_rho[j];
                const int cnt = g_counts[j];
                X.rho[j] = rho;
                X.cntv[j] = cnt;
                value_view2(j, x, a.no_vnorm ? -1.0f / (float)cnt : rho, sm);
            }
        } else {
            // slots not founded yet: zero direction (S = 0) and zero read view
            const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                if (!vside) {
                    *reinterpret_cast<uint4*>(sm + OFF_UHI + swz(j, ch)) = z;
                    *reinterpret_cast<uint4*>(sm + OFF_ULO + swz(j, ch)) = z;
                    *reinterpret_cast<uint4*>(sm + OFF_VK + swz(j, ch)) = z;
                } else {
                    *reinterpret_cast<uint4*>(sm + OFF_VV + swz(j, ch)) = z;
                }
            }
        }
    }
    tc_fence_before();
    fence_proxy_async();
    __syncthreads();
    tc_fence_after();

    const uint32_t idesc = idesc_bf16(128, 256, 0, 0);
    int mma_count = 0;
    // S = k (u_hi + u_lo)^T for the 128 chunk keys in buffer b against all 256 slot directions
    auto issue_mma = [&](int b) {
        tc_fence_after();
        for (int ks = 0; ks < 4; ++ks)
            for (int part = 0; part < 2; ++part) {
                const uint64_t ad = sdesc_sw128(sK + b * TOK * ROWB + ks * 32, 16, 1024);
                const uint64_t bd = sdesc_sw128((part ? sUL : sUH) + ks * 32, 16, 1024);
                mma_bf16_ss(tmem + 256, ad, bd, idesc, (ks | part) ? 1u : 0u);
            }
        mma_commit(bar_s);
        pend_mma = mma_count & 1;
    };
    KVM_PROBE_DECL(20)
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
        // every thread waits for the chunk itself (nothing of the previous event is
        // read after its last barrier, so the set-up below needs no barrier first);
        // a failed wait is carried to the next barrier, which all threads leave together
        bool fail = !mbar_wait(smem_u32(&X.bar_k[buf]), (it >> 1) & 1, &X.abort_flag, a.status);
        if (!fail) pend_ld[buf] = -1;
        if (e + 1 < a.e_end) {
            sc_nx = a.sched ? a.sched[e + 1] : a.sched0;
            if (tid < C) g_nx = a.g_src[(int64_t)bh * a.src_row + ((int64_t)(e + 1) * C) % a.src_len + tid];
        }
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
        // the first event of a launch: thread 0 issues its MMA; every later one was issued
        // at the end of the previous event by the issuer warp
        if (tid == 0 && !fail && do_mma && it == 0) issue_mma(buf);
        if (tid < C) X.g[tid] = g_here;
        // per-token set-up: two threads per token (warps 8-15), 32 dims each
        if (vside) {
            const int t = (tid - MAXS) >> 1, h = tid & 1;
            float ss = t < C ? sq_row_sw<4>(kch, t, 4 * h) : 0.0f;
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);
            if (t < C && h == 0) {
                X.kn[t] = sqrtf(ss);
                const bool sink = first_pos + t < S;
                X.kind[t] = sink ? 2 : -1;
                X.slot[t] = sink ? (int)(first_pos + t) : -1;
            }
        } else {
            X.slot_tok[j] = -1;
            *reinterpret_cast<uint4*>(&X.tmask[j][0]) = make_uint4(0, 0, 0, 0);
        }
        KVM_PROBE_LAP(1)

        // best / second / argmax over the mergeable slots [S, n0): each quarter of
        // the CTA scans 64 slot columns of every token row (token = TMEM lane)
        if (do_mma) {
            fail = fail || !mbar_wait(bar_s, mma_count & 1, &X.abort_flag, a.status);
            if (!fail) pend_mma = -1;
            KVM_PROBE_LAP(9)
            ++mma_count;
            tc_fence_after();
            const int q = tid >> 7, t = tid & 127;
            const int lo = max(S, q * 64), hi = min(n0, q * 64 + 64);
            float b0 = -INFINITY, s0 = -INFINITY, b1 = -INFINITY, s1 = -INFINITY;
            int a0 = -1, a1 = -1;
            if (lo < hi && !__any_sync(0xffffffffu, fail)) {
                uint32_t va[32], vb[32];
                tmem_ld32(t_sim + q * 64, va);
                tmem_ld32(t_sim + q * 64 + 32, vb);
                tmem_wait_ld();
                KVM_PROBE_LAP(11)
                scan32<GAP>(va, q * 64, lo, hi, b0, s0, a0);
                scan32<GAP>(vb, q * 64 + 32, lo, hi, b1, s1, a1);
            }
            merge_later(b0, s0, a0, b1, s1, a1);
            KVM_PROBE_LAP(12)
            X.pb[q][t] = b0;
            X.ps[q][t] = s0;
            X.pa[q][t] = a0;
            tc_fence_before();
        }
        if (__syncthreads_or(fail)) break;
        KVM_PROBE_LAP(2)
        float best = -INFINITY, sec = -INFINITY;
        int barg = -1;
        const bool cand = tid < C && X.kind[tid] != 2;
        if (cand && do_mma) {
#pragma unroll
            for (int q = 0; q < 4; ++q) merge_later(best, sec, barg, X.pb[q][tid], X.ps[q][tid], X.pa[q][tid]);
        }
        const float kn = tid < C ? X.kn[tid] : 0.0f;
        if (cand) X.m[tid] = barg < 0 ? -INFINITY : (kn > 0.0f ? best / kn : 0.0f);
        // events that append slots or found sinks exchange per-token results; the
        // others (every token merges) touch only their own token's entries until
        // the merge lists below
        const bool slow = na > 0 || first_pos < S;
        if (slow) __syncthreads();

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
        if (slow) {
            __syncthreads();
            if (tid < C && X.kind[tid] != 0) X.slot_tok[X.slot[tid]] = tid;
            __syncthreads();
        }
        KVM_PROBE_LAP(3)

        if (na > 0) {
            // directions of the new slots (from their founding token), then the
            // remaining tokens also compare against them
            if (!vside && j >= n0 && j < n0 + na) {
                const int t = X.slot_tok[j];
                float kx[64];
                set_row_sw(kch, t, X.g[t], kx);
                const float mean = sum64(kx) * (1.0f / 64.0f);
#pragma unroll
                for (int x = 0; x < 64; ++x) kx[x] -= mean;
                const float ss = dot64(kx, kx);
                const float inv = ss > 0.0f ? 1.0f / sqrtf(ss) : 0.0f;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    uint32_t hw[4], lw[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float a0 = kx[ch * 8 + 2 * u] * inv;
                        const float a1 = kx[ch * 8 + 2 * u + 1] * inv;
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
                set_row_sw(kch, tid, 1.0f, kx);
                for (int jj = n0; jj < n0 + na; ++jj) {
                    // k . (u_hi + u_lo), partial sums by dim mod 8 in dim order
                    float p[8];
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        const uint4 hw = *reinterpret_cast<const uint4*>(sm + OFF_UHI + swz(jj, ch));
                        const uint4 lw = *reinterpret_cast<const uint4*>(sm + OFF_ULO + swz(jj, ch));
                        const uint32_t hv[4] = {hw.x, hw.y, hw.z, hw.w}, lv[4] = {lw.x, lw.y, lw.z, lw.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const float2 hf = bf2(hv[u]), lf = bf2(lv[u]);
                            const float u0 = hf.x + lf.x, u1 = hf.y + lf.y;
                            if (ch == 0) {
                                p[2 * u] = kx[2 * u] * u0;
                                p[2 * u + 1] = kx[2 * u + 1] * u1;
                            } else {
                                p[2 * u] = fmaf(kx[ch * 8 + 2 * u], u0, p[2 * u]);
                                p[2 * u + 1] = fmaf(kx[ch * 8 + 2 * u + 1], u1, p[2 * u + 1]);
                            }
                        }
                    }
                    const float s = ((p[0] + p[1]) + (p[2] + p[3])) + ((p[4] + p[5]) + (p[6] + p[7]));
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
            if (GAP && a.dbg_gap) {
                float gp = __int_as_float(0x7fc00000);
                if (kd == 0) gp = sec == -INFINITY ? INFINITY : (kn > 0.0f ? (best - sec) / kn : 0.0f);
                a.dbg_gap[o] = gp;
            }
        }

        KVM_PROBE_LAP(4)
        // merge lists: each merged token sets its bit in its slot's 128-bit token mask
        // (OR commutes, so the masks do not depend on timing); an owner then visits
        // its tokens in position order, lowest bit first
        if (tid < C && X.kind[tid] == 0 && X.slot[tid] >= 0 &&
            kvm_check(X.slot[tid] >= S && X.slot[tid] < sc.n_after, a.status))
            atomicOr(&X.tmask[X.slot[tid]][tid >> 5], 1u << (tid & 31));
        // the previous snapshot store must have finished reading the view
        if (tid == TMA_T) bulk_wait_read();
        __syncthreads();
        KVM_PROBE_LAP(5)

        // owners: founding and merging into their slot (key owner: key sums and
        // count; value owner: value sums and read radius), then the new read view
        {
            const int ft = X.slot_tok[j];
            const uint4 mk = *reinterpret_cast<const uint4*>(&X.tmask[j][0]);
            const int nm = __popc(mk.x) + __popc(mk.y) + __popc(mk.z) + __popc(mk.w);
            const bool touched = ft >= 0 || nm > 0;
            const bool wtouched = __any_sync(0xffffffffu, touched);
            float2 x[32];
            int cnt = 0;
            float ss = 0.0f;

            if (wtouched) {
                const uint8_t* rows = vside ? vch : kch;
                tmem_ld64_2(t_own, x);
                KVM_PROBE_LAP(18)
                float rho = 0.0f;
                if (touched) {
                    if (!vside) cnt = X.cnt[j];
                    else {
                        rho = X.rho[j];
                        cnt = X.cntv[j];
                    }
                    if (ft >= 0) {
                        set_row_sw2(rows, ft, X.g[ft], x);
                        cnt = 0;
                        if (vside) rho = sqrtf(sq_row_sw<8>(vch, ft, 0));
                    }
                    // merged tokens in position order, one loop over the whole 128-bit mask
                    // (a warp runs as many rounds as its busiest slot has tokens)
                    unsigned long long m_lo = ((unsigned long long)mk.y << 32) | mk.x;
                    unsigned long long m_hi = ((unsigned long long)mk.w << 32) | mk.z;
                    while (m_lo | m_hi) {
                        const bool low = m_lo != 0ull;
                        const unsigned long long m = low ? m_lo : m_hi;
                        const int t = (low ? 0 : 64) + __ffsll((long long)m) - 1;
                        if (low) m_lo &= m_lo - 1; else m_hi &= m_hi - 1;
                        add_row_sw2(rows, t, X.g[t], x);
                    }
                    cnt += nm + (ft >= 0 ? 1 : 0);
                }
                KVM_PROBE_LAP(13)
                tmem_st64_2(t_own, x);
                tmem_wait_st();
                KVM_PROBE_LAP(14)
                if (touched) {
                    if (!vside) {
                        X.cnt[j] = cnt;
                        ss = key_dir2(j, x, sm);
                        // the next event's MMA reads these directions (async proxy)
                        fence_proxy_async();
                        KVM_PROBE_LAP(15)
                        key_view2(j, x, ss, cnt, a.r, a.ln_eps, sm);
                        KVM_PROBE_LAP(19)
                    } else {
                        X.rho[j] = rho;
                        X.cntv[j] = cnt;
                        value_view2(j, x, a.no_vnorm ? -1.0f / (float)cnt : rho, sm);
                    }
                }
            }
            if (!vside || warp == MMA_W) {
                // every direction of this event is written (and fenced by its writer): the
                // issuer warp (its own read views written and fenced first) issues the next
                // event's similarity MMA now, while the value owners finish
                if (warp == MMA_W) fence_proxy_async();
                KVM_PROBE_LAP(16)
                asm volatile("bar.sync 1, 288;" ::: "memory");
                KVM_PROBE_LAP(17)
                if (tid == MMA_W * 32 && e + 1 < a.e_end && !X.abort_flag && sc_nx.n0 > S) {
                    if (mbar_wait(smem_u32(&X.bar_k[buf ^ 1]), ((it + 1) >> 1) & 1, &X.abort_flag, a.status))
                        issue_mma(buf ^ 1);
                }
            }
        }
        KVM_PROBE_LAP(6)
        tc_fence_before();
        fence_proxy_async();
        // the event's closing barrier: every warp but the issuer (which met the key side
        // above after its last access of this event's chunk and state rows)
        if (warp != MMA_W) asm volatile("bar.sync 2, 480;" ::: "memory");
        tc_fence_after();

        // chunk e + 2 loads into this event's buffer (its readers passed the barrier
        // above), ahead of the snapshot copies in the copy engine's queue
        if (tid == TMA_T && e + 2 < a.e_end) load_chunk(e + 2, buf);
        // snapshot of the read view after this event (async bulk copy)
        if (tid == TMA_T && a.snap_k && e < a.snap_events) {
            // the swizzled view rows leave by TMA tensor stores (the copy engine unswizzles)
            const int plane = bh * a.snap_events + e;
            tma_store_3d(&tm_snk, smem_u32(sm + OFF_VK), 0, 0, plane);
            tma_store_3d(&tm_snv, smem_u32(sm + OFF_VV), 0, 0, plane);
            bulk_commit();
        }
        n = sc.n_after;
        KVM_PROBE_LAP(7)
    }
    // the issuer warp left the last event without its closing barrier: every warp is done
    // with the chunk area (the value sums' staging tiles below) before anyone writes there
    __syncthreads();

    // write the state back for decode, export and later segments: the sums go
    // through swizzled staging tiles (key sums in the direction area, value sums
    // in the chunk area) and leave by TMA; the read view leaves by bulk copy
    if (tid == TMA_T) bulk_wait_all();
    {
        float x[64];
        tmem_ld64(t_own, x);
        uint8_t* stage = sm + (vside ? OFF_K : OFF_UHI);
#pragma unroll
        for (int q = 0; q < 16; ++q)
            *reinterpret_cast<float4*>(stage + stage_off(j, q)) =
                make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
        if (j < n && !X.abort_flag) {
            if (!vside) g_counts[j] = X.cnt[j];
            else g_rho[j] = X.rho[j];
        }
    }
    fence_proxy_async();
    __syncthreads();
    // the compact read-key view (the non-rotary 16-byte pieces of every row) leaves by
    // plain stores; the read-value view and the sums by TMA
    if (n > 0 && !X.abort_flag) {
        const int DK = view_k_dims(a.r), zc = (D - DK) / 8, pr = DK / 8;
        uint4* gvk = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.view_k) + (int64_t)bh * M * DK);
        for (int i = tid; i < n * pr; i += NT) {
            const int row = i / pr, pc = zc + (i - row * pr);
            gvk[i] = *reinterpret_cast<const uint4*>(sm + OFF_VK + swz(row, pc));
        }
    }
    if (tid == TMA_T && n > 0 && !X.abort_flag) {
        const int nb = (n + srows - 1) / srows;
        for (int h = 0; h < 2; ++h)
            for (int b = 0; b < nb; ++b) {
                const uint32_t o = h * 32768 + b * srows * 128;
                tma_store_3d(&tm_sk, smem_u32(sm + OFF_UHI) + o, 32 * h, b * srows, bh);
                tma_store_3d(&tm_sv, smem_u32(sm + OFF_K) + o, 32 * h, b * srows, bh);
            }
        tma_store_3d(&tm_vv, smem_u32(sm + OFF_VV), 0, 0, bh);
        bulk_commit();
        bulk_wait_all();
    }
    KVM_PROBE_LAP(10)
    if (tid == 0 || tid == 255 || tid == 256 || tid == 511)
        KVM_PROBE_FLUSH(g_probe_fold, 20 * (tid == 0 ? 0 : tid == 255 ? 1 : tid == 256 ? 2 : 3), 20)
    // after an abort: let the copies and MMAs this CTA issued land before its shared
    // and tensor memory are released (each wait bounded; they depend on nothing else)
    if (X.abort_flag && (tid == 0 || tid == TMA_T || tid == MMA_W * 32)) {
        auto drain = [&](uint32_t bar, int parity) {
            if (parity < 0) return;
            const long long t0 = clock64();
            while (!mbar_try(bar, (uint32_t)parity) && clock64() - t0 < (1ll << 28)) {
            }
        };
        if (tid == 0 || tid == MMA_W * 32) {
            if (tid == 0) drain(smem_u32(&X.bar_st), pend_st);
            drain(bar_s, pend_mma);
        } else {
            drain(smem_u32(&X.bar_k[0]), pend_ld[0]);
            drain(smem_u32(&X.bar_k[1]), pend_ld[1]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace foldtc

KVM_PROBE_READOUT(kvm_probe_read_fold, foldtc::g_probe_fold)

bool fold_tc_supported(const FoldArgs& a, bool bf16) { return bf16 && a.C <= 128 && a.M <= foldtc::MAXS; }

cudaError_t launch_fold_tc(const FoldArgs& args, cudaStream_t s) {
    FoldArgs a = args;
    a.stage_rows = a.M < foldtc::STAGE_ROWS ? a.M : foldtc::STAGE_ROWS;
    CUtensorMap mk, mv, msk, msv, msnk, msnv, mvv;
    // read-value view: [BH][M][64] bf16 stored a whole state (M <= 256 rows) per box;
    // snapshots [BH * events][M][64] (maps of the read-value view when there are none:
    // nothing is stored through them then)
    const bool snaps = a.snap_k && a.snap_events > 0;
    const uint64_t snap_planes = snaps ? (uint64_t)a.BH * a.snap_events : (uint64_t)a.BH;
    if (!make_tmap_bf16_3d(&mk, a.k_src, (uint64_t)a.src_row, (uint64_t)a.BH, 128) ||
        !make_tmap_bf16_3d(&mv, a.v_src, (uint64_t)a.src_row, (uint64_t)a.BH, 128) ||
        !make_tmap_f32_3d(&msk, a.sum_k, (uint64_t)a.M, (uint64_t)a.BH, (uint32_t)a.stage_rows) ||
        !make_tmap_f32_3d(&msv, a.sum_v, (uint64_t)a.M, (uint64_t)a.BH, (uint32_t)a.stage_rows) ||
        !make_tmap_bf16_3d(&mvv, a.view_v, (uint64_t)a.M, (uint64_t)a.BH, (uint32_t)a.M) ||
        !make_tmap_bf16_3d(&msnk, snaps ? a.snap_k : a.view_v, (uint64_t)a.M, snap_planes, (uint32_t)a.M) ||
        !make_tmap_bf16_3d(&msnv, snaps ? a.snap_v : a.view_v, (uint64_t)a.M, snap_planes, (uint32_t)a.M))
        return cudaErrorInvalidValue;
    // the second-best similarity is tracked only when the debug record wants the top-2 gap
    auto kern = a.dbg_gap ? foldtc::fold_tc_kernel<true> : foldtc::fold_tc_kernel<false>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, foldtc::SMEM_BYTES);
    kern<<<a.BH, foldtc::NT, foldtc::SMEM_BYTES, s>>>(mk, mv, msk, msv, msnk, msnv, mvv, a);
    return cudaGetLastError();
}

}  // namespace kvm
