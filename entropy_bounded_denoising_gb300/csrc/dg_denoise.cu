// dg_denoise.cu -- the denoise step: per-position statistics and sampling (K1), per-canvas
// acceptance / renoise / convergence (K2), canvas initialisation and loop bookkeeping.
//
// Method (DiffusionGemma vLLM page, "DiffusionGemma: vLLM이 네이티브로 지원하는 최초의 디퓨전
// 언어 모델(dLLM)"): section "엔트로피 기반 디노이징" (entropy H(p) = -sum p log p, the
// entropy-bound acceptance rule, the convergence rule) and section
// "DiffusionGemmaModelState와 DiffusionSampler" (Denoise case: logits / T, Gumbel-max
// candidates argmax(logits / T + g), acceptance up to the entropy bound, renoise of the
// rest, argmax canvas, convergence check; Prefill case: random canvas).  Read-only
// canvases follow the single-pass-reads page ("답은 한 번 읽는데 모델은 왜 두 번 돌까?"):
// one pass, statistics only.
//
// K1 design (GB300): one thread-block cluster per canvas position.  Each CTA pulls its
// slice of the logit row into shared memory with bulk copies (TMA engine) in pieces, so the
// row is read from HBM exactly once; pass A folds the slice into an online-softmax state
// (max m, count c of entries equal to m, r = sum of the other e^z, t = sum e^z z) -- the
// split keeps near-one-hot rows accurate in fp32 -- plus the argmax; CTAs merge through
// distributed shared memory in rank order (a reduction tree fixed by V alone, so a row's
// result does not depend on the batch it came in).  Pass B draws the Gumbel noise only for
// entries that can still win: an entry with z + G_max below the best score so far cannot,
// and a cheap bound on u rejects most of the rest before the two logarithms.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <math.h>

#include "dg_common.cuh"

namespace cg = cooperative_groups;

namespace {

constexpr int kK1Threads = 256;
constexpr int kK1Warps = kK1Threads / 32;
constexpr int kMaxPieces = 8;
constexpr int kMaxCluster = 8;
constexpr uint32_t kMaxChunkBytes = 192u * 1024u;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Largest Gumbel value the uniform mapping can produce, -log(-log(1 - 2^-24)) = 16.6355...,
// rounded up; plus a margin for the candidate test.
constexpr float kGumbelMax = 16.64f;
constexpr float kCandidateSlack = 1e-3f;
// Exponents (log2 units) below this give 2^d = 0 in fp32 with flush-to-zero.
constexpr float kMinExponent = -256.f;

struct RowState {  // online softmax state of a set of entries, z measured in log2 units
    float m;       // max raw logit (-inf = empty)
    float c;       // entries equal to m
    float r;       // sum of 2^d over the other entries, d = (x - m) * log2e / T
    float t;       // sum of 2^d * d
    int idx;       // smallest index attaining m
};

struct K1Shared {
    uint64_t bar[kMaxPieces];
    RowState warp_state[kK1Warps];
    RowState cta_state;  // read by the other CTAs of the cluster
    RowState row_state;
    float warp_best[kK1Warps];
    int warp_bidx[kK1Warps];
    float cta_best;  // read by the other CTAs of the cluster
    int cta_bidx;
    int bad;
    int timeout;
};

DG_DEVINL float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// max that keeps a NaN operand (so NaN logits still poison the row state)
DG_DEVINL float max_nan(float a, float b) {
    float y;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
    return y;
}

// Merge two states; k2 = log2e / T.  Sides whose max is below the new max are rescaled and
// their max entries join r.
DG_DEVINL RowState merge(RowState a, RowState b, float k2) {
    if (b.m == -INFINITY && b.c == 0.f && b.r == 0.f) return a;
    if (a.m == -INFINITY && a.c == 0.f && a.r == 0.f) return b;
    const float M = fmaxf(a.m, b.m);
    RowState o;
    o.m = M;
    o.idx = (a.m > b.m) ? a.idx : (b.m > a.m) ? b.idx : min(a.idx, b.idx);
    if (a.m < M) {
        const float d = (a.m - M) * k2, al = ex2(d), s = a.c + a.r;
        a.t = al * (a.t + d * s);
        a.r = al * s;
        a.c = 0.f;
    }
    if (b.m < M) {
        const float d = (b.m - M) * k2, al = ex2(d), s = b.c + b.r;
        b.t = al * (b.t + d * s);
        b.r = al * s;
        b.c = 0.f;
    }
    o.c = a.c + b.c;
    o.r = a.r + b.r;
    o.t = a.t + b.t;
    return o;
}

DG_DEVINL RowState shfl_state(RowState s, int lane_mask) {
    RowState o;
    o.m = __shfl_xor_sync(0xffffffffu, s.m, lane_mask);
    o.c = __shfl_xor_sync(0xffffffffu, s.c, lane_mask);
    o.r = __shfl_xor_sync(0xffffffffu, s.r, lane_mask);
    o.t = __shfl_xor_sync(0xffffffffu, s.t, lane_mask);
    o.idx = __shfl_xor_sync(0xffffffffu, s.idx, lane_mask);
    return o;
}

DG_DEVINL bool better(float s, int i, float bs, int bi) { return s > bs || (s == bs && i < bi); }

template <int DT>
struct Vec;  // 16 bytes of logits as floats

template <>
struct Vec<0> {  // bf16: 8 entries
    static constexpr int N = 8;
    DG_DEVINL static void load(const unsigned char* p, float (&x)[8]) {
        const uint4 q = *reinterpret_cast<const uint4*>(p);
        x[0] = __uint_as_float(q.x << 16);
        x[1] = __uint_as_float(q.x & 0xffff0000u);
        x[2] = __uint_as_float(q.y << 16);
        x[3] = __uint_as_float(q.y & 0xffff0000u);
        x[4] = __uint_as_float(q.z << 16);
        x[5] = __uint_as_float(q.z & 0xffff0000u);
        x[6] = __uint_as_float(q.w << 16);
        x[7] = __uint_as_float(q.w & 0xffff0000u);
    }
};

template <>
struct Vec<1> {  // fp32: 4 entries
    static constexpr int N = 4;
    DG_DEVINL static void load(const unsigned char* p, float (&x)[4]) {
        const float4 q = *reinterpret_cast<const float4*>(p);
        x[0] = q.x;
        x[1] = q.y;
        x[2] = q.z;
        x[3] = q.w;
    }
};

// ------------------------------------------------------------------------------------
// K1: per-position statistics and Gumbel-max sample.  grid (CS, L, n), cluster (CS, 1, 1).
// ------------------------------------------------------------------------------------
template <int DT>
__global__ void __launch_bounds__(kK1Threads) k1_row_stats(
    const unsigned char* __restrict__ logits, int64_t ld_bytes, int64_t V, int32_t L,
    const dg_canvas_params* __restrict__ params, uint64_t seed, int32_t chunk_elems,
    int32_t* __restrict__ argmax_out, int32_t* __restrict__ sample_out, float* __restrict__ entropy_out,
    float* __restrict__ lse_out, unsigned* status) {
    constexpr int VN = Vec<DT>::N;
    constexpr int ES = DT == 0 ? 2 : 4;
    extern __shared__ __align__(128) unsigned char k1_smem[];
    K1Shared& sh = *reinterpret_cast<K1Shared*>(k1_smem);
    unsigned char* chunk = k1_smem + ((sizeof(K1Shared) + 127) / 128) * 128;

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int ncta = (int)cluster.num_blocks();
    const int pos = blockIdx.y;
    const int64_t canvas = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    const dg_canvas_params p = params[canvas];
    if (!(p.flags & DG_ACTIVE)) return;  // whole cluster leaves together
    if (!(p.temperature > 0.f) || !isfinite(p.temperature)) {
        if (rank == 0 && tid == 0 && pos == 0) dg::raise_status(status, DG_DEV_BAD_PARAM);
        return;
    }
    const bool do_sample = !(p.flags & DG_READ_ONLY);
    const float invT = 1.0f / p.temperature;
    const float k2 = kLog2e * invT;

    const int64_t row = canvas * L + pos;
    const int64_t begin = (int64_t)rank * chunk_elems;
    const int64_t end = min(V, begin + (int64_t)chunk_elems);
    const int n_el = (int)max((int64_t)0, end - begin);
    const uint32_t bytes = (uint32_t)n_el * ES;
    const uint32_t bulk = bytes & ~15u;
    const int nvec = (n_el + VN - 1) / VN;
    const unsigned char* src = logits + row * ld_bytes + begin * ES;

    int npieces = (int)((bytes + 8191u) / 8192u);
    npieces = max(1, min(kMaxPieces, npieces));
    const int vpp = (nvec + npieces - 1) / npieces;

    if (tid == 0) {
        for (int i = 0; i < npieces; ++i) dg::mbar_init(&sh.bar[i], 1);
        dg::fence_mbar_init();
        sh.bad = 0;
        sh.timeout = 0;
    }
    __syncthreads();
    if (tid == 0) {
        for (int i = 0; i < npieces; ++i) {
            const uint32_t lo = (uint32_t)min(nvec, i * vpp) * 16u;
            const uint32_t hi = min(bulk, (uint32_t)min(nvec, (i + 1) * vpp) * 16u);
            if (hi > lo) {
                dg::mbar_arrive_expect_tx(&sh.bar[i], hi - lo);
                dg::bulk_g2s(chunk + lo, src + lo, hi - lo, &sh.bar[i]);
            } else {
                dg::mbar_arrive(&sh.bar[i]);
            }
        }
    }
    // ragged tail (< 16 bytes) by plain loads
    if (tid < (int)(bytes - bulk)) chunk[bulk + tid] = src[bulk + tid];
    __syncthreads();

    // ---------------- pass A: online softmax state and argmax
    RowState st{-INFINITY, 0.f, 0.f, 0.f, 0x7fffffff};
    bool bad = false;
    for (int pc = 0; pc < npieces; ++pc) {
        if (!dg::mbar_wait(&sh.bar[pc], 0)) {
            sh.timeout = 1;
            break;
        }
        const int vlo = pc * vpp, vhi = min(nvec, vlo + vpp);
        for (int j = vlo + tid; j < vhi; j += kK1Threads) {
            float x[VN];
            Vec<DT>::load(chunk + (size_t)j * 16, x);
            const int base = j * VN;
            if (base + VN > n_el) {
#pragma unroll
                for (int i = 0; i < VN; ++i)
                    if (base + i >= n_el) x[i] = -INFINITY;
            }
            float vmax = x[0];
#pragma unroll
            for (int i = 1; i < VN; ++i) vmax = fmaxf(vmax, x[i]);
            if (vmax > st.m) {
                int i0 = VN - 1;
#pragma unroll
                for (int i = VN - 1; i >= 0; --i)
                    if (x[i] == vmax) i0 = i;
                if (st.m == -INFINITY) {
                    st.c = 0.f;
                    st.r = 0.f;
                    st.t = 0.f;
                } else {
                    const float d = (st.m - vmax) * k2, al = ex2(d), s = st.c + st.r;
                    st.t = al * (st.t + d * s);
                    st.r = al * s;
                    st.c = 0.f;
                }
                st.m = vmax;
                st.idx = (int)begin + base + i0;
            }
            if (vmax == st.m) {
                if (vmax == -INFINITY) {
#pragma unroll
                    for (int i = 0; i < VN; ++i) bad |= (x[i] != x[i]);
                    continue;
                }
#pragma unroll
                for (int i = 0; i < VN; ++i) {
                    if (x[i] == st.m) {
                        st.c += 1.f;
                    } else {
                        // -inf entries (masked tail, or -inf logits) contribute e = 0; the clamp
                        // keeps e * d at 0 instead of 0 * -inf
                        const float d = max_nan((x[i] - st.m) * k2, kMinExponent), e = ex2(d);
                        st.r += e;
                        st.t = fmaf(e, d, st.t);
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < VN; ++i) {
                    const float d = max_nan((x[i] - st.m) * k2, kMinExponent), e = ex2(d);
                    st.r += e;
                    st.t = fmaf(e, d, st.t);
                }
            }
        }
    }
    if (bad) sh.bad = 1;

    // warp, CTA and cluster merges (fixed order)
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) st = merge(st, shfl_state(st, o), k2);
    if (lane == 0) sh.warp_state[warp] = st;
    __syncthreads();
    if (tid == 0) {
        RowState c = sh.warp_state[0];
        for (int w = 1; w < kK1Warps; ++w) c = merge(c, sh.warp_state[w], k2);
        sh.cta_state = c;
    }
    cluster.sync();
    if (tid == 0) {
        RowState rs = *cluster.map_shared_rank(&sh.cta_state, 0);
        for (int q = 1; q < ncta; ++q) rs = merge(rs, *cluster.map_shared_rank(&sh.cta_state, q), k2);
        int any_bad = 0;
        for (int q = 0; q < ncta; ++q) any_bad |= cluster.map_shared_rank(&sh.bad, q)[0];
        sh.row_state = rs;
        sh.bad = any_bad;
    }
    __syncthreads();
    const RowState rs = sh.row_state;
    const bool empty = rs.m == -INFINITY;
    const bool row_bad = sh.bad || rs.m == INFINITY || !isfinite(rs.r) || !isfinite(rs.t);

    // ---------------- pass B: Gumbel-max over entries that can still win
    float best = -INFINITY;
    int bidx = 0x7fffffff;
    const uint32_t k0 = (uint32_t)seed, k1 = p.request_id;
    const uint32_t c3 = dg::ctr_word3(seed, dg::kStreamGumbel);
    const uint32_t step = (uint32_t)p.step;
    if (do_sample && !empty && !row_bad && !sh.timeout) {
        {  // the argmax entry gives the first lower bound (z = 0 there)
            const dg::u4 w = dg::philox10((uint32_t)rs.idx >> 2, (uint32_t)pos, step, c3, k0, k1);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
            const float u = dg::uniform_from_word(ws[rs.idx & 3]);
            best = 0.f + (-logf(-logf(u)));
            bidx = rs.idx;
        }
        for (int j = tid; j < nvec; j += kK1Threads) {
            float x[VN];
            Vec<DT>::load(chunk + (size_t)j * 16, x);
            const int base = j * VN;
#pragma unroll
            for (int h = 0; h < VN; h += 4) {
                float z[4];
                bool any = false;
                const float thr = best - kGumbelMax - kCandidateSlack;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float xi = (base + h + i < n_el) ? x[h + i] : -INFINITY;
                    z[i] = (xi - rs.m) * invT;
                    any |= (z[i] >= thr);
                }
                if (!any) continue;
                const int v0 = (int)begin + base + h;  // multiple of 4
                const dg::u4 w = dg::philox10((uint32_t)v0 >> 2, (uint32_t)pos, step, c3, k0, k1);
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (!(z[i] >= best - kGumbelMax - kCandidateSlack)) continue;
                    const float u = dg::uniform_from_word(ws[i]);
                    // g > D = best - z needs u > exp(-e^-D) >= 1 - e^-D; keep a factor 2 of slack
                    const float eb = 2.f * ex2(-(best - z[i]) * kLog2e);
                    if (!(u > 1.f - eb)) continue;
                    const float score = z[i] + (-logf(-logf(u)));
                    if (better(score, v0 + i, best, bidx)) {
                        best = score;
                        bidx = v0 + i;
                    }
                }
            }
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const float ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
        if (better(ob, oi, best, bidx)) {
            best = ob;
            bidx = oi;
        }
    }
    if (lane == 0) {
        sh.warp_best[warp] = best;
        sh.warp_bidx[warp] = bidx;
    }
    __syncthreads();
    if (tid == 0) {
        float b = sh.warp_best[0];
        int bi = sh.warp_bidx[0];
        for (int w = 1; w < kK1Warps; ++w)
            if (better(sh.warp_best[w], sh.warp_bidx[w], b, bi)) {
                b = sh.warp_best[w];
                bi = sh.warp_bidx[w];
            }
        sh.cta_best = b;
        sh.cta_bidx = bi;
    }
    cluster.sync();
    if (rank == 0 && tid == 0) {
        float b = sh.cta_best;
        int bi = sh.cta_bidx;
        int any_timeout = sh.timeout;
        for (int q = 1; q < ncta; ++q) {
            const float ob = *cluster.map_shared_rank(&sh.cta_best, q);
            const int oi = *cluster.map_shared_rank(&sh.cta_bidx, q);
            any_timeout |= *cluster.map_shared_rank(&sh.timeout, q);
            if (better(ob, oi, b, bi)) {
                b = ob;
                bi = oi;
            }
        }
        // H = log(c + r) - t ln2 / (c + r), with log1p where a single entry holds the max
        const float s = rs.c + rs.r;
        const float lns = (rs.c == 1.f) ? log1pf(rs.r) : logf(rs.c) + log1pf(rs.r / rs.c);
        const float H = lns - rs.t * kLn2 / s;
        entropy_out[row] = H;
        lse_out[row] = rs.m * invT + lns;
        argmax_out[row] = empty ? 0 : rs.idx;
        sample_out[row] = (do_sample && !empty && !row_bad) ? bi : -1;
        if (row_bad) dg::raise_status(status, DG_DEV_NAN_INF_ROW);
        if (empty) dg::raise_status(status, DG_DEV_EMPTY_ROW);
        if (any_timeout) dg::raise_status(status, DG_DEV_TIMEOUT);
    }
    // keep every CTA's shared memory alive until the peers are done reading it, and make
    // sure no bulk copy is still landing when the CTA exits
    if (sh.timeout && tid == 0)
        for (int pc = 0; pc < npieces; ++pc) (void)dg::mbar_wait(&sh.bar[pc], 0);
    cluster.sync();
}

// ------------------------------------------------------------------------------------
// K2: acceptance, renoise and convergence for one canvas per CTA (blockDim = 32 * ceil(L/32)).
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) k2_accept(
    const float* __restrict__ entropy, const int32_t* __restrict__ sample, const int32_t* __restrict__ argmax,
    int32_t L, int64_t V, const dg_canvas_params* __restrict__ params, uint64_t seed, int32_t* __restrict__ canvas,
    int32_t* __restrict__ prev_argmax, int32_t* __restrict__ stable_count, uint8_t* __restrict__ accept_mask,
    uint8_t* __restrict__ converged, float* __restrict__ mean_entropy, int32_t* __restrict__ n_accept,
    unsigned* status) {
    __shared__ float sH[1024];
    __shared__ double sSorted[1024];
    __shared__ double sWarp[32];
    __shared__ int sCut;

    const int64_t c = blockIdx.x;
    const int i = threadIdx.x, lane = i & 31, warp = i >> 5, nwarps = blockDim.x >> 5;
    const dg_canvas_params p = params[c];
    if (!(p.flags & DG_ACTIVE)) return;
    if (!(p.temperature > 0.f) || !isfinite(p.temperature) || p.k < 1 || p.max_steps < 1 || p.min_accept < 0 ||
        p.min_accept > L) {
        if (i == 0) dg::raise_status(status, DG_DEV_BAD_PARAM);
        return;
    }
    const bool read_only = (p.flags & DG_READ_ONLY) != 0;
    const bool valid = i < L;
    const int64_t q = c * L + i;
    const float H = valid ? entropy[q] : 0.f;
    const int32_t am = valid ? argmax[q] : 0;
    if (valid) sH[i] = H;
    if (i == 0) sCut = L;
    __syncthreads();

    // rank in (entropy, position) order
    int rk = 0;
    if (valid) {
        for (int j = 0; j < L; ++j) {
            const float hj = sH[j];
            rk += (hj < H) || (hj == H && j < i);
        }
        sSorted[rk] = (double)H;
    }
    __syncthreads();

    // inclusive prefix sums of the sorted entropies (fp64)
    double v = valid ? sSorted[i] : 0.0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) sWarp[warp] = v;
    __syncthreads();
    if (warp == 0) {
        double w = lane < nwarps ? sWarp[lane] : 0.0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double n = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += n;
        }
        sWarp[lane] = w;
    }
    __syncthreads();
    if (warp > 0) v += sWarp[warp - 1];
    // the first sorted position whose running sum exceeds beta ends the accepted prefix
    if (valid && v > (double)p.beta) atomicMin(&sCut, i);
    const double Hsum = sWarp[nwarps - 1];
    __syncthreads();

    int nacc = max(p.min_accept, sCut);
    nacc = min(nacc, L);
    if (read_only) nacc = 0;

    const bool same = __syncthreads_and(!valid || am == prev_argmax[q]) != 0;
    if (valid) {
        const bool acc = rk < nacc;
        accept_mask[q] = acc ? 1 : 0;
        if (!read_only)
            canvas[q] = acc ? sample[q]
                            : (int32_t)dg::random_token(seed, p.request_id, (uint32_t)p.step, (uint32_t)i,
                                                        dg::kStreamRenoise, (uint32_t)V);
        prev_argmax[q] = am;
    }
    if (i == 0) {
        const int32_t st = same ? stable_count[c] + 1 : 0;
        const double Hbar = Hsum / (double)L;
        bool conv = (st >= p.k && Hbar < (double)p.tau) || (p.step + 1 >= p.max_steps);
        if (read_only) conv = true;
        stable_count[c] = st;
        converged[c] = conv ? 1 : 0;
        if (mean_entropy) mean_entropy[c] = (float)Hbar;
        if (n_accept) n_accept[c] = nacc;
    }
}

__global__ void k_canvas_init(int32_t* __restrict__ canvas, int32_t L, int64_t V,
                              const dg_canvas_params* __restrict__ params, uint64_t seed) {
    const int64_t c = blockIdx.x;
    const dg_canvas_params p = params[c];
    if (!(p.flags & DG_ACTIVE)) return;
    for (int i = threadIdx.x; i < L; i += blockDim.x)
        canvas[c * L + i] = (int32_t)dg::random_token(seed, p.request_id, (uint32_t)p.step, (uint32_t)i,
                                                      dg::kStreamInit, (uint32_t)V);
}

__global__ void k_advance_params(dg_canvas_params* __restrict__ params, const uint8_t* __restrict__ converged,
                                 int64_t n) {
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= n) return;
    dg_canvas_params p = params[c];
    if (!(p.flags & DG_ACTIVE)) return;
    if (converged[c]) p.flags &= ~(uint32_t)DG_ACTIVE;
    else p.step += 1;
    params[c] = p;
}

__global__ void k_philox_words(uint64_t seed, uint32_t request_id, uint32_t step, uint32_t position, uint32_t sid,
                               uint32_t block0, int64_t n_blocks, uint32_t* __restrict__ out) {
    const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= n_blocks) return;
    const dg::u4 w =
        dg::philox10(block0 + (uint32_t)b, position, step, dg::ctr_word3(seed, sid), (uint32_t)seed, request_id);
    reinterpret_cast<uint4*>(out)[b] = make_uint4(w.x, w.y, w.z, w.w);
}

// ------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

dg_status check_canvas_dims(int64_t n, int32_t L, int64_t V) {
    if (n < 0 || n > 65535 || L < 1 || L > 1024 || V < 2 || V > 0x7fffffffLL) return DG_ERR_INVALID_ARG;
    return DG_OK;
}

struct K1Plan {
    int cs;
    int32_t chunk_elems;
    size_t smem;
};

bool plan_k1(dg_dtype dt, int64_t V, K1Plan* pl) {
    const int64_t es = dt == DG_BF16 ? 2 : 4;
    const int64_t vn = 16 / es;
    const int64_t row_bytes = V * es;
    int cs = 1;
    while (cs < kMaxCluster && row_bytes > (int64_t)cs * 65536) cs *= 2;
    int64_t chunk = (V + cs - 1) / cs;
    chunk = (chunk + vn - 1) / vn * vn;
    if (chunk * es > (int64_t)kMaxChunkBytes) return false;
    pl->cs = cs;
    pl->chunk_elems = (int32_t)chunk;
    pl->smem = ((sizeof(K1Shared) + 127) / 128) * 128 + (size_t)((chunk * es + 127) / 128 * 128);
    return true;
}

template <int DT>
dg_status launch_k1(const void* logits, int64_t ld, int64_t n, int32_t L, int64_t V,
                    const dg_canvas_params* params, uint64_t seed, const K1Plan& pl, int32_t* argmax, int32_t* sample,
                    float* entropy, float* lse, cudaStream_t stream) {
    auto kern = k1_row_stats<DT>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pl.smem) != cudaSuccess)
        return DG_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)pl.cs, (unsigned)L, (unsigned)n);
    cfg.blockDim = dim3(kK1Threads, 1, 1);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)pl.cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int64_t ld_bytes = ld * (DT == 0 ? 2 : 4);
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<const unsigned char*>(logits), ld_bytes, V, L, params,
                                       seed, pl.chunk_elems, argmax, sample, entropy, lse, dghost::status_word());
    dghost::count_launch();
    return dghost::cuda_status(e);
}

dg_status launch_k2(const float* entropy, const int32_t* sample, const int32_t* argmax, int64_t n, int32_t L,
                    int64_t V, const dg_canvas_params* params, uint64_t seed, int32_t* canvas, int32_t* prev_argmax,
                    int32_t* stable_count, uint8_t* accept_mask, uint8_t* converged, float* mean_entropy,
                    int32_t* n_accept, cudaStream_t stream) {
    const unsigned threads = (unsigned)((L + 31) / 32 * 32);
    k2_accept<<<(unsigned)n, threads, 0, stream>>>(entropy, sample, argmax, L, V, params, seed, canvas, prev_argmax,
                                                   stable_count, accept_mask, converged, mean_entropy, n_accept,
                                                   dghost::status_word());
    dghost::count_launch();
    return dghost::cuda_status(cudaGetLastError());
}

}  // namespace

extern "C" {

size_t dg_denoise_workspace_bytes(int64_t, int32_t, int64_t, dg_dtype) { return 0; }

dg_status dg_denoise_step(const void* logits, dg_dtype dtype, int64_t ld, int64_t n_canvas, int32_t L, int64_t V,
                          const dg_canvas_params* params, uint64_t seed, int32_t* canvas, int32_t* prev_argmax,
                          int32_t* stable_count, uint8_t* accept_mask, int32_t* argmax, int32_t* sample,
                          float* entropy, float* lse, uint8_t* converged, float* mean_entropy, int32_t* n_accept,
                          void* workspace, size_t workspace_bytes, dg_stream_t stream) {
    (void)workspace;
    (void)workspace_bytes;
    if (dtype != DG_BF16 && dtype != DG_FP32) return DG_ERR_INVALID_ARG;
    dg_status s = check_canvas_dims(n_canvas, L, V);
    if (s != DG_OK) return s;
    if (ld < V) return DG_ERR_INVALID_ARG;
    if (n_canvas == 0) return DG_OK;
    if (!logits || !params || !canvas || !prev_argmax || !stable_count || !accept_mask || !argmax || !sample ||
        !entropy || !lse || !converged)
        return DG_ERR_INVALID_ARG;
    const int64_t es = dtype == DG_BF16 ? 2 : 4;
    if (!aligned16(logits) || (ld * es) % 16 != 0) return DG_ERR_ALIGNMENT;
    K1Plan pl;
    if (!plan_k1(dtype, V, &pl)) return DG_ERR_UNSUPPORTED;
    cudaStream_t st = (cudaStream_t)stream;
    s = dtype == DG_BF16 ? launch_k1<0>(logits, ld, n_canvas, L, V, params, seed, pl, argmax, sample, entropy, lse, st)
                         : launch_k1<1>(logits, ld, n_canvas, L, V, params, seed, pl, argmax, sample, entropy, lse, st);
    if (s != DG_OK) return s;
    return launch_k2(entropy, sample, argmax, n_canvas, L, V, params, seed, canvas, prev_argmax, stable_count,
                     accept_mask, converged, mean_entropy, n_accept, st);
}

dg_status dg_accept_from_entropy(const float* entropy, const int32_t* sample, const int32_t* argmax,
                                 int64_t n_canvas, int32_t L, int64_t V, const dg_canvas_params* params,
                                 uint64_t seed, int32_t* canvas, int32_t* prev_argmax, int32_t* stable_count,
                                 uint8_t* accept_mask, uint8_t* converged, float* mean_entropy, int32_t* n_accept,
                                 dg_stream_t stream) {
    dg_status s = check_canvas_dims(n_canvas, L, V);
    if (s != DG_OK) return s;
    if (n_canvas == 0) return DG_OK;
    if (!entropy || !sample || !argmax || !params || !canvas || !prev_argmax || !stable_count || !accept_mask ||
        !converged)
        return DG_ERR_INVALID_ARG;
    return launch_k2(entropy, sample, argmax, n_canvas, L, V, params, seed, canvas, prev_argmax, stable_count,
                     accept_mask, converged, mean_entropy, n_accept, (cudaStream_t)stream);
}

dg_status dg_canvas_init(int32_t* canvas, int64_t n_canvas, int32_t L, int64_t V, const dg_canvas_params* params,
                         uint64_t seed, dg_stream_t stream) {
    dg_status s = check_canvas_dims(n_canvas, L, V);
    if (s != DG_OK) return s;
    if (n_canvas == 0) return DG_OK;
    if (!canvas || !params) return DG_ERR_INVALID_ARG;
    k_canvas_init<<<(unsigned)n_canvas, 256, 0, (cudaStream_t)stream>>>(canvas, L, V, params, seed);
    dghost::count_launch();
    return dghost::cuda_status(cudaGetLastError());
}

dg_status dg_advance_params(dg_canvas_params* params, const uint8_t* converged, int64_t n_canvas,
                            dg_stream_t stream) {
    if (n_canvas < 0) return DG_ERR_INVALID_ARG;
    if (n_canvas == 0) return DG_OK;
    if (!params || !converged) return DG_ERR_INVALID_ARG;
    const unsigned blocks = (unsigned)((n_canvas + 255) / 256);
    k_advance_params<<<blocks, 256, 0, (cudaStream_t)stream>>>(params, converged, n_canvas);
    dghost::count_launch();
    return dghost::cuda_status(cudaGetLastError());
}

dg_status dg_philox_words(uint64_t seed, uint32_t request_id, uint32_t step, uint32_t position, uint32_t stream_id,
                          uint32_t block0, int64_t n_blocks, uint32_t* out, dg_stream_t stream) {
    if (n_blocks < 0 || stream_id > 255u) return DG_ERR_INVALID_ARG;
    if (n_blocks == 0) return DG_OK;
    if (!out) return DG_ERR_INVALID_ARG;
    if (!aligned16(out)) return DG_ERR_ALIGNMENT;
    const int64_t blocks = (n_blocks + 255) / 256;
    if (blocks > 0x7fffffffLL) return DG_ERR_INVALID_ARG;
    k_philox_words<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(seed, request_id, step, position, stream_id,
                                                                       block0, n_blocks, out);
    dghost::count_launch();
    return dghost::cuda_status(cudaGetLastError());
}

}  // extern "C"
