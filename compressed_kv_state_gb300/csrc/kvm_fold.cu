// Fold chain of the KVM layer: the sequential per-(batch, head) state update
// (the portable chain, for fp32 layers; bf16 layers use the tensor-core chains).
//
// "Key-Value Means" (gist.science technical summary):
//   Core mechanism 1 - a chunk that overflows the window is folded into the
//                      state, not dropped;
//   Core mechanism 2 - winner-take-all merge into the slot whose LayerNorm'd
//                      key has the highest cosine with the token's key; the
//                      gate scales what is absorbed; values are read at the
//                      slot's read radius;
//   Core mechanism 3 - the most surprising tokens become new slots;
//   Core mechanism 5 - protected sink rows;
//   lay part "smart merge" - raw sums and counts, divided only when read.
//
// One CTA owns one (b,h) row and runs its events back to back; the state
// lives in the workspace (L2-resident at these sizes).  Every step is a
// block-wide phase separated by __syncthreads.  The merge is deterministic:
// merged tokens are sorted by (slot, position) and each (slot, dim) pair is
// accumulated by one thread in position order, so no atomics are used.
#include "kvm_internal.cuh"

namespace kvm {

constexpr int FOLD_THREADS = 256;
constexpr int UTILE = 32;  // slot directions staged per shared-memory tile

// Recompute the read view and the similarity direction of slot j (one warp).
template <typename T>
__device__ __forceinline__ void renorm_slot(const float* sk, const float* sv, int cnt, float rho,
                                            float* sd, T* vk, T* vv, int r, float eps, int lane,
                                            int no_vnorm) {
    float s0 = sk[lane], s1 = sk[lane + 32];
    // similarity direction: unit(s - mean(s)); the cosine against LayerNorm(s / count)
    // equals the cosine against this (LayerNorm centres and scales only)
    float mean = warp_sum(s0 + s1) * (1.0f / D);
    float c0 = s0 - mean, c1 = s1 - mean;
    float ss = warp_sum(c0 * c0 + c1 * c1);
    float inv = ss > 0.0f ? 1.0f / sqrtf(ss) : 0.0f;
    if (sizeof(T) == 2) {
        // bf16 layers: the row holds the direction as bf16 hi + lo terms (elements
        // [0, 64) and [64, 128)), the form the tensor-core fold chains stream
        __nv_bfloat16* u = reinterpret_cast<__nv_bfloat16*>(sd);
        const float a0 = c0 * inv, a1 = c1 * inv;
        const __nv_bfloat16 h0 = __float2bfloat16_rn(a0), h1 = __float2bfloat16_rn(a1);
        u[lane] = h0;
        u[lane + 32] = h1;
        u[64 + lane] = __float2bfloat16_rn(a0 - __bfloat162float(h0));
        u[64 + lane + 32] = __float2bfloat16_rn(a1 - __bfloat162float(h1));
    } else {
        sd[lane] = c0 * inv;
        sd[lane + 32] = c1 * inv;
    }
    // read key: LayerNorm(s / count), no affine, biased variance, rotary dims zeroed
    float ic = 1.0f / (float)cnt;
    float x0 = s0 * ic, x1 = s1 * ic;
    float mx = warp_sum(x0 + x1) * (1.0f / D);
    float d0 = x0 - mx, d1 = x1 - mx;
    float var = warp_sum(d0 * d0 + d1 * d1) * (1.0f / D);
    float rs = 1.0f / sqrtf(var + eps);
    // vk holds dims [D - view_k_dims(r), D) of the read key (the compact view)
    const int k0 = D - view_k_dims(r);
    if (lane >= k0) vk[lane - k0] = from_f<T>(lane < r ? 0.0f : d0 * rs);
    if (lane + 32 >= k0) vk[lane + 32 - k0] = from_f<T>(lane + 32 < r ? 0.0f : d1 * rs);
    // read value: rho * unit(sum_v) (ablation: the member mean sum_v / count)
    float v0 = sv[lane], v1 = sv[lane + 32];
    float nv = sqrtf(warp_sum(v0 * v0 + v1 * v1));
    float f = no_vnorm ? ic : (nv > 0.0f ? rho / nv : 0.0f);
    vv[lane] = from_f<T>(v0 * f);
    vv[lane + 32] = from_f<T>(v1 * f);
}

// Two CTAs per SM (at most 128 registers a thread, no spills): a fold at a decode
// step's chunk boundary runs one CTA for each of up to thousands of (b, h) rows.
template <typename T>
__global__ void __launch_bounds__(FOLD_THREADS, 2) fold_chain_kernel(FoldArgs a) {
    extern __shared__ float4 smem4[];
    float* smem = reinterpret_cast<float*>(smem4);
    const int C = a.C, S = a.S, M = a.M;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = FOLD_THREADS / 32;
    const int bh = blockIdx.x;

    float* kf = smem;                   // [C][D] chunk keys, fp32
    float* vf = kf + C * D;             // [C][D] chunk values
    float* ut = vf + C * D;             // [UTILE][D] staged slot directions
    float* gs = ut + UTILE * D;         // [C] gates
    float* kn = gs + C;                 // [C] key norms
    float* ms = kn + C;                 // [C] surprise score
    float* bd = ms + C;                 // [C] best dot
    float* sdt = bd + C;                // [C] second-best dot
    int* kind = reinterpret_cast<int*>(sdt + C);  // [C] 0 merged, 1 appended, 2 sink, -1 none
    int* slot = kind + C;               // [C] destination slot
    int* sorted = slot + C;             // [C] merged tokens sorted by (slot, pos)
    int* seg = sorted + C;              // [C + 1] segment starts
    int* touched = seg + C + 1;         // [C] slots to renormalise
    __shared__ int sh_cnt[4];

    float* sum_k = a.sum_k + (int64_t)bh * M * D;
    float* sum_v = a.sum_v + (int64_t)bh * M * D;
    int* counts = a.counts + (int64_t)bh * M;
    float* rho = a.rho + (int64_t)bh * M;
    float* simdir = a.simdir + (int64_t)bh * M * D;
    const int DK = view_k_dims(a.r);  // dims of a compact read-key row
    T* view_k = reinterpret_cast<T*>(a.view_k) + (int64_t)bh * M * DK;
    T* view_v = reinterpret_cast<T*>(a.view_v) + (int64_t)bh * M * D;
    const T* ksrc = reinterpret_cast<const T*>(a.k_src) + (int64_t)bh * a.src_row * D;
    const T* vsrc = reinterpret_cast<const T*>(a.v_src) + (int64_t)bh * a.src_row * D;
    const float* gsrc = a.g_src + (int64_t)bh * a.src_row;

    for (int e = a.e_begin; e < a.e_end; ++e) {
        const Sched sc = a.sched ? a.sched[e] : a.sched0;
        const int64_t first_pos = (int64_t)e * C;
        const int64_t off = first_pos % a.src_len;

        // 1. stage the chunk (keys, values, gates) and the key norms
        for (int i = tid; i < C * D; i += FOLD_THREADS) {
            kf[i] = to_f<T>(ksrc[off * D + i]);
            vf[i] = to_f<T>(vsrc[off * D + i]);
        }
        for (int i = tid; i < C; i += FOLD_THREADS) gs[i] = gsrc[off + i];
        __syncthreads();
        for (int t = warp; t < C; t += nwarps) {
            float x0 = kf[t * D + lane], x1 = kf[t * D + lane + 32];
            float nn = warp_sum(x0 * x0 + x1 * x1);
            if (lane == 0) {
                kn[t] = sqrtf(nn);
                kind[t] = (first_pos + t < S) ? 2 : -1;
            }
        }
        __syncthreads();

        // 2. sinks: the first S tokens of the sequence found slots 0..S-1
        for (int t = warp; t < C; t += nwarps) {
            if (kind[t] != 2) continue;
            const int j = (int)(first_pos + t);
            const float g = gs[t];
            sum_k[j * D + lane] = g * kf[t * D + lane];
            sum_k[j * D + lane + 32] = g * kf[t * D + lane + 32];
            sum_v[j * D + lane] = g * vf[t * D + lane];
            sum_v[j * D + lane + 32] = g * vf[t * D + lane + 32];
            float v0 = vf[t * D + lane], v1 = vf[t * D + lane + 32];
            float nv = sqrtf(warp_sum(v0 * v0 + v1 * v1));
            if (lane == 0) {
                counts[j] = 1;
                rho[j] = nv;
                slot[t] = j;
            }
        }

        // 3. surprise: best cosine of each candidate against the mergeable slots [S, n0)
        const int n0 = sc.n0;
        const bool cand_thread = tid < C;
        float kr[D];
        if (cand_thread) {
#pragma unroll
            for (int x = 0; x < D; ++x) kr[x] = kf[tid * D + x];
        }
        float best = -INFINITY, second = -INFINITY;
        int barg = -1;
        for (int j0 = S; j0 < n0; j0 += UTILE) {
            const int cnt = min(UTILE, n0 - j0);
            __syncthreads();
            for (int i = tid; i < cnt * D; i += FOLD_THREADS) ut[i] = simdir[(int64_t)j0 * D + i];
            __syncthreads();
            if (cand_thread && kind[tid] != 2) {
                for (int jj = 0; jj < cnt; ++jj) {
                    float s = 0.0f;
#pragma unroll
                    for (int x = 0; x < D; ++x) s = fmaf(kr[x], ut[jj * D + x], s);
                    if (s > best) {
                        second = best;
                        best = s;
                        barg = j0 + jj;
                    } else if (s > second) {
                        second = s;
                    }
                }
            }
        }
        if (cand_thread && kind[tid] != 2) {
            const float nk = kn[tid];
            ms[tid] = (barg < 0) ? -INFINITY : (nk > 0.0f ? best / nk : 0.0f);
        }
        __syncthreads();

        // 4. choose the a most surprising candidates (smallest score, then lowest position)
        const int na = sc.a;
        int rank = 0;
        const bool is_cand = cand_thread && kind[tid] != 2;
        if (is_cand) {
            const float mt = ms[tid];
            for (int u = 0; u < C; ++u) {
                if (kind[u] == 2) continue;
                const float mu = ms[u];
                rank += (mu < mt) || (mu == mt && u < tid);
            }
        }
        __syncthreads();
        if (is_cand) kind[tid] = rank < na ? 1 : 0;
        __syncthreads();
        // appended slots in position order
        if (cand_thread && kind[tid] == 1) {
            int before = 0;
            for (int u = 0; u < tid; ++u) before += (kind[u] == 1);
            slot[tid] = n0 + before;
        }
        __syncthreads();

        // 5. found the appended slots: sums g*k, g*v, count 1, rho = |v|
        for (int t = warp; t < C; t += nwarps) {
            if (kind[t] != 1) continue;
            const int j = slot[t];
            const float g = gs[t];
            sum_k[j * D + lane] = g * kf[t * D + lane];
            sum_k[j * D + lane + 32] = g * kf[t * D + lane + 32];
            sum_v[j * D + lane] = g * vf[t * D + lane];
            sum_v[j * D + lane + 32] = g * vf[t * D + lane + 32];
            float v0 = vf[t * D + lane], v1 = vf[t * D + lane + 32];
            float nv = sqrtf(warp_sum(v0 * v0 + v1 * v1));
            float s0 = g * kf[t * D + lane], s1 = g * kf[t * D + lane + 32];
            float mean = warp_sum(s0 + s1) * (1.0f / D);
            float c0 = s0 - mean, c1 = s1 - mean;
            float ss = warp_sum(c0 * c0 + c1 * c1);
            float inv = ss > 0.0f ? 1.0f / sqrtf(ss) : 0.0f;
            simdir[j * D + lane] = c0 * inv;
            simdir[j * D + lane + 32] = c1 * inv;
            if (lane == 0) {
                counts[j] = 1;
                rho[j] = nv;
            }
        }

        // 6. the remaining candidates also see the new slots [n0, n0 + a)
        for (int j0 = n0; j0 < n0 + na; j0 += UTILE) {
            const int cnt = min(UTILE, n0 + na - j0);
            __syncthreads();
            for (int i = tid; i < cnt * D; i += FOLD_THREADS) ut[i] = simdir[(int64_t)j0 * D + i];
            __syncthreads();
            if (cand_thread && kind[tid] == 0) {
                for (int jj = 0; jj < cnt; ++jj) {
                    float s = 0.0f;
#pragma unroll
                    for (int x = 0; x < D; ++x) s = fmaf(kr[x], ut[jj * D + x], s);
                    if (s > best) {
                        second = best;
                        best = s;
                        barg = j0 + jj;
                    } else if (s > second) {
                        second = s;
                    }
                }
            }
        }
        if (cand_thread && kind[tid] == 0) {
            slot[tid] = barg;
            if (barg < 0 && a.status) atomicOr(a.status, STATUS_DEVICE);
            const float nk = kn[tid];
            bd[tid] = nk > 0.0f ? best / nk : 0.0f;
            sdt[tid] = second == -INFINITY ? -INFINITY : (nk > 0.0f ? second / nk : 0.0f);
        }
        __syncthreads();

        // debug record
        if (cand_thread && e < a.dbg_events) {
            const int64_t o = ((int64_t)bh * a.dbg_events + e) * C + tid;
            const int kd = kind[tid];
            if (a.dbg_assign) a.dbg_assign[o] = slot[tid];
            if (a.dbg_kind) a.dbg_kind[o] = kd;
            if (a.dbg_m) a.dbg_m[o] = kd == 2 ? __int_as_float(0x7fc00000) : ms[tid];
            if (a.dbg_gap) {
                float gp = __int_as_float(0x7fc00000);
                if (kd == 0) gp = sdt[tid] == -INFINITY ? INFINITY : bd[tid] - sdt[tid];
                a.dbg_gap[o] = gp;
            }
        }

        // 7. merge: sort merged tokens by (slot, position), one owner per (slot, dim)
        if (cand_thread && kind[tid] == 0) {
            const int mj = slot[tid];
            int rank = 0;
            for (int u = 0; u < C; ++u) {
                if (kind[u] != 0) continue;
                const int su = slot[u];
                rank += (su < mj) || (su == mj && u < tid);
            }
            sorted[rank] = tid;
        }
        if (tid == 0) {
            int nm = 0;
            for (int u = 0; u < C; ++u) nm += (kind[u] == 0);
            sh_cnt[0] = nm;
        }
        __syncthreads();
        const int nmerged = sh_cnt[0];
        if (tid < nmerged) {
            const bool head = tid == 0 || slot[sorted[tid]] != slot[sorted[tid - 1]];
            if (head) {
                int before = 0;
                for (int i = 1; i <= tid; ++i) before += (slot[sorted[i]] != slot[sorted[i - 1]]);
                seg[before] = tid;
            }
        }
        if (tid == 0) {
            int ns = 0;
            for (int i = 0; i < nmerged; ++i) ns += (i == 0 || slot[sorted[i]] != slot[sorted[i - 1]]);
            sh_cnt[1] = ns;
            seg[ns] = nmerged;
        }
        __syncthreads();
        const int nseg = sh_cnt[1];
        for (int pidx = tid; pidx < nseg * 2 * D; pidx += FOLD_THREADS) {
            const int sgi = pidx / (2 * D);
            const int rem = pidx - sgi * 2 * D;
            const bool isv = rem >= D;
            const int x = isv ? rem - D : rem;
            const int beg = seg[sgi], end = seg[sgi + 1];
            const int j = slot[sorted[beg]];
            float* dst = (isv ? sum_v : sum_k) + (int64_t)j * D + x;
            const float* src = isv ? vf : kf;
            float acc = *dst;
            for (int i = beg; i < end; ++i) {
                const int tok = sorted[i];
                acc = fmaf(gs[tok], src[tok * D + x], acc);
            }
            *dst = acc;
        }
        for (int sgi = tid; sgi < nseg; sgi += FOLD_THREADS) {
            const int j = slot[sorted[seg[sgi]]];
            counts[j] += seg[sgi + 1] - seg[sgi];
            touched[sgi] = j;
        }
        __syncthreads();
        // sinks and appended slots are touched too
        if (tid == 0) {
            int nt = nseg;
            for (int t = 0; t < C; ++t)
                if (kind[t] == 1 || kind[t] == 2) touched[nt++] = slot[t];
            sh_cnt[2] = nt;
        }
        __syncthreads();

        // 8. just-in-time read view of the touched slots
        const int ntouch = sh_cnt[2];
        for (int i = warp; i < ntouch; i += nwarps) {
            const int j = touched[i];
            renorm_slot<T>(sum_k + (int64_t)j * D, sum_v + (int64_t)j * D, counts[j], rho[j],
                           simdir + (int64_t)j * D, view_k + (int64_t)j * DK,
                           view_v + (int64_t)j * D, a.r, a.ln_eps, lane, a.no_vnorm);
        }
        __syncthreads();

        // 9. snapshot of the view after this event, for the attention of chunk e + W/C + 1
        if (a.snap_k && e < a.snap_events) {
            // full snapshot rows: the compact key view's rows behind zeros on the
            // leading dims it does not store
            const int64_t base = ((int64_t)bh * a.snap_events + e) * M * D;
            constexpr int CPR = D * (int)sizeof(T) / 16;     // 16-byte pieces of a full row
            const int zc = (D - DK) * (int)sizeof(T) / 16;   // pieces before the compact part
            const int n_pc = sc.n_after * CPR;
            const uint4* sk4 = reinterpret_cast<const uint4*>(view_k);
            const uint4* sv4 = reinterpret_cast<const uint4*>(view_v);
            uint4* dk4 = reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.snap_k) + base);
            uint4* dv4 = reinterpret_cast<uint4*>(reinterpret_cast<T*>(a.snap_v) + base);
            for (int i = tid; i < n_pc; i += FOLD_THREADS) {
                const int row = i / CPR, pc = i - row * CPR;
                dk4[i] = pc < zc ? make_uint4(0u, 0u, 0u, 0u) : sk4[row * (CPR - zc) + pc - zc];
                dv4[i] = sv4[i];
            }
        }
        __syncthreads();
    }
}

// Recompute simdir and the read view of slots [0, n) of every row (state import).
template <typename T>
__global__ void renorm_all_kernel(RenormArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t total = (int64_t)a.BH * a.n;
    if (gw >= total) return;
    const int64_t bh = gw / a.n, j = gw % a.n;
    const int64_t row = bh * a.M + j;
    if (!kvm_check(a.counts[row] >= 1, a.status)) return;
    renorm_slot<T>(a.sum_k + row * D, a.sum_v + row * D, a.counts[row], a.rho[row],
                   a.simdir + row * D, reinterpret_cast<T*>(a.view_k) + row * view_k_dims(a.r),
                   reinterpret_cast<T*>(a.view_v) + row * D, a.r, a.ln_eps, lane, a.no_vnorm);
}

static size_t fold_smem_bytes(int C) {
    return sizeof(float) * ((size_t)2 * C * D + UTILE * D + 5 * C) + sizeof(int) * (5 * (size_t)C + 1);
}

cudaError_t launch_fold(const FoldArgs& a, bool bf16, cudaStream_t s) {
    // bf16 layers fold on the tensor cores (the state on chip up to 256 slots and
    // 128 tokens a chunk, else streamed); this portable chain serves fp32 layers
    if (fold_tc_supported(a, bf16)) return launch_fold_tc(a, s);
    if (fold_big_supported(a, bf16)) return launch_fold_big(a, s);
    if (bf16) return cudaErrorInvalidValue;
    const size_t smem = fold_smem_bytes(a.C);
    cudaFuncSetAttribute(fold_chain_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    fold_chain_kernel<float><<<a.BH, FOLD_THREADS, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_renorm(const RenormArgs& a, bool bf16, cudaStream_t s) {
    const int64_t warps = (int64_t)a.BH * a.n;
    if (warps == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = (warps * 32 + threads - 1) / threads;
    if (bf16)
        renorm_all_kernel<__nv_bfloat16><<<(unsigned)blocks, threads, 0, s>>>(a);
    else
        renorm_all_kernel<float><<<(unsigned)blocks, threads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace kvm
