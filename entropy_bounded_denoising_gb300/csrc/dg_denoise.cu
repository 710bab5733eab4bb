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
// K1 design (GB300): one CTA per canvas position streams its logit row once from HBM.  A
// producer warp keeps a ring of shared-memory slots filled with bulk copies (the TMA
// engine); eight consumer warps fold every piece into an online-softmax state (max m,
// count c of entries equal to m, r = sum of the other e^z, t = sum e^z z -- the split keeps
// near-one-hot rows accurate in fp32) and the argmax, and in the same pass look for the
// Gumbel-max winner: an entry whose y + G_max (G_max the largest Gumbel value the uniform
// mapping can produce) cannot reach the best score seen so far in the CTA is skipped
// without drawing its noise; the others are queued per warp and drawn 32 groups at a time.
// The reduction order depends only on V, so a row's result does not depend on its batch.
#include <cuda_runtime.h>

#include <math.h>

#include "dg_common.cuh"

namespace {

constexpr int kK1Warps = 8;                        // consumer warps
constexpr int kK1Threads = (kK1Warps + 1) * 32;    // + one producer warp
constexpr int kSlots = 4;                          // ring of shared-memory slots
constexpr uint32_t kPieceBytes = 16384;            // bytes per slot
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

template <int DT>
struct K1Shared {
    static constexpr int kQW = DT == 0 ? 2 : 4;  // words per queued group (4 bf16 or 4 fp32)
    uint64_t full[kSlots];
    uint64_t empty[kSlots];
    RowState warp_state[kK1Warps];
    float warp_best[kK1Warps];
    int warp_bidx[kK1Warps];
    unsigned best_key;  // CTA-wide best score so far, order-preserving integer encoding
    int bad;
    int timeout;
    // per-warp candidate groups awaiting their Gumbel draw: first entry index and the 4
    // logits (as raw words), so a queued group outlives the ring slot it came from
    int q_e0[kK1Warps][96];
    uint32_t q_x[kK1Warps][96][kQW];
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

// Float <-> unsigned keys with the same order (for atomicMax on scores).
DG_DEVINL unsigned float_key(float f) {
    const unsigned b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
DG_DEVINL float key_float(unsigned k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
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

DG_DEVINL uint32_t word_of(const dg::u4& w, int i) {
    return i == 0 ? w.x : i == 1 ? w.y : i == 2 ? w.z : w.w;
}

DG_DEVINL void warp_best(float& best, int& bidx) {
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const float ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
        if (better(ob, oi, best, bidx)) {
            best = ob;
            bidx = oi;
        }
    }
}

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

// Gumbel draw for one group of 4 consecutive entries (one Philox block) [e0, e0 + 4) with
// logits x.  Keeps (best, bidx) as the largest score y + g, y = x / T, ties to the lower
// index.  `bound` is a score some entry of the row is known to reach; entries that cannot
// reach it are not drawn.
DG_DEVINL void eval_group(const float (&x)[4], int e0, int64_t V, float invT, uint32_t pos, uint32_t step,
                          uint32_t c3, uint32_t k0, uint32_t k1, float bound, float& best, int& bidx) {
    const dg::u4 w = dg::philox10((uint32_t)e0 >> 2, pos, step, c3, k0, k1);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (e0 + i >= V) continue;
        const float y = x[i] * invT;
        const float b = fmaxf(bound, best);
        if (!(y >= b - kGumbelMax - kCandidateSlack)) continue;
        const float u = dg::uniform_from_word(word_of(w, i));
        // g > D = b - y needs u > exp(-e^-D) >= 1 - e^-D; keep a factor 2 of slack
        const float eb = 2.f * ex2(-(b - y) * kLog2e);
        if (!(u > 1.f - eb)) continue;
        const float score = y + (-logf(-logf(u)));
        if (better(score, e0 + i, best, bidx)) {
            best = score;
            bidx = e0 + i;
        }
    }
}

// Raw words <-> 4 logits of a group (bf16 pairs or fp32).
template <int DT, int N>
DG_DEVINL void group_words(const float (&x)[N], int g, uint32_t (&w)[4]) {
    if (DT == 0) {
        w[0] = (__float_as_uint(x[4 * g]) >> 16) | (__float_as_uint(x[4 * g + 1]) & 0xffff0000u);
        w[1] = (__float_as_uint(x[4 * g + 2]) >> 16) | (__float_as_uint(x[4 * g + 3]) & 0xffff0000u);
        w[2] = 0u;
        w[3] = 0u;
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = __float_as_uint(x[4 * g + i]);
    }
}

template <int DT>
DG_DEVINL void words_group(const uint32_t* w, float (&x)[4]) {
    if (DT == 0) {
        x[0] = __uint_as_float(w[0] << 16);
        x[1] = __uint_as_float(w[0] & 0xffff0000u);
        x[2] = __uint_as_float(w[1] << 16);
        x[3] = __uint_as_float(w[1] & 0xffff0000u);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = __uint_as_float(w[i]);
    }
}

// ------------------------------------------------------------------------------------
// K1: per-position statistics and Gumbel-max sample.  grid (L, n), one CTA per position.
// ------------------------------------------------------------------------------------
template <int DT>
__global__ void __launch_bounds__(kK1Threads, 3) k1_row_stats(
    const unsigned char* __restrict__ logits, int64_t ld_bytes, int64_t V, int32_t L,
    const dg_canvas_params* __restrict__ params, uint64_t seed, int32_t* __restrict__ argmax_out,
    int32_t* __restrict__ sample_out, float* __restrict__ entropy_out, float* __restrict__ lse_out,
    unsigned* status) {
    constexpr int VN = Vec<DT>::N;
    constexpr int ES = DT == 0 ? 2 : 4;
    constexpr int GPV = VN / 4;                    // Philox blocks per 16-byte vector
    constexpr int kPieceElems = kPieceBytes / ES;
    extern __shared__ __align__(128) unsigned char k1_smem[];
    using Shared = K1Shared<DT>;
    constexpr int QW = Shared::kQW;
    Shared& sh = *reinterpret_cast<Shared*>(k1_smem);
    unsigned char* ring = k1_smem + ((sizeof(Shared) + 127) / 128) * 128;

    const int pos = blockIdx.x;
    const int64_t canvas = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    const dg_canvas_params p = params[canvas];
    if (!(p.flags & DG_ACTIVE)) return;
    if (!(p.temperature > 0.f) || !isfinite(p.temperature)) {
        if (tid == 0 && pos == 0) dg::raise_status(status, DG_DEV_BAD_PARAM);
        return;
    }
    const bool do_sample = !(p.flags & DG_READ_ONLY);
    const float invT = 1.0f / p.temperature;
    const float k2 = kLog2e * invT;
    const int64_t row = canvas * L + pos;
    const unsigned char* src = logits + row * ld_bytes;
    const uint32_t bytes = (uint32_t)(V * ES);
    const uint32_t bulk = bytes & ~15u;
    const int npieces = (int)((bytes + kPieceBytes - 1) / kPieceBytes);

    if (tid == 0) {
        for (int i = 0; i < kSlots; ++i) {
            dg::mbar_init(&sh.full[i], 1);
            dg::mbar_init(&sh.empty[i], kK1Warps);
        }
        dg::fence_mbar_init();
        sh.bad = 0;
        sh.timeout = 0;
        sh.best_key = float_key(-INFINITY);
    }
    __syncthreads();

    if (warp == kK1Warps) {
        // ---------------- producer: keep the ring full
        if (lane == 0) {
            for (int q = 0; q < npieces; ++q) {
                const int sl = q % kSlots;
                if (q >= kSlots && !dg::mbar_wait(&sh.empty[sl], (uint32_t)((q / kSlots) - 1) & 1u)) {
                    sh.timeout = 1;
                    break;
                }
                unsigned char* dst = ring + (size_t)sl * kPieceBytes;
                const uint32_t lo = (uint32_t)q * kPieceBytes;
                const uint32_t hi = min(bytes, lo + kPieceBytes);
                const uint32_t bhi = min(bulk, hi);
                // the ragged tail (< 16 bytes) by plain copies, ordered before the arrive below
                for (uint32_t b = max(bulk, lo); b < hi; ++b) dst[b - lo] = src[b];
                dg::mbar_arrive_expect_tx(&sh.full[sl], bhi > lo ? bhi - lo : 0u);
                if (bhi > lo) dg::bulk_g2s(dst, src + lo, bhi - lo, &sh.full[sl]);
            }
            if (sh.timeout) {  // never leave with a copy still landing in shared memory
                for (int i = 0; i < kSlots; ++i) (void)dg::mbar_wait(&sh.full[i], 0);
                for (int i = 0; i < kSlots; ++i) (void)dg::mbar_wait(&sh.full[i], 1);
            }
        }
    } else {
        // ---------------- consumers
        RowState st{-INFINITY, 0.f, 0.f, 0.f, 0x7fffffff};
        bool bad = false;
        float best = -INFINITY;    // this warp's best score and its entry
        int bidx = 0x7fffffff;
        float bound = -INFINITY;   // best score known anywhere in the CTA
        const uint32_t k0 = (uint32_t)seed, k1 = p.request_id;
        const uint32_t c3 = dg::ctr_word3(seed, dg::kStreamGumbel);
        const uint32_t step = (uint32_t)p.step;
        int* q_e0 = sh.q_e0[warp];
        uint32_t(*q_x)[QW] = sh.q_x[warp];
        int qn = 0;  // warp-uniform queue length, kept across pieces
        const unsigned lt = (1u << lane) - 1u;
        for (int q = 0; q < npieces; ++q) {
            const int sl = q % kSlots;
            if (!dg::mbar_wait(&sh.full[sl], (uint32_t)(q / kSlots) & 1u)) {
                sh.timeout = 1;
                break;
            }
            const unsigned char* slot = ring + (size_t)sl * kPieceBytes;
            const int e_lo = q * kPieceElems;
            const int n_el = (int)min((int64_t)kPieceElems, V - e_lo);
            const int nvec = (n_el + VN - 1) / VN;
            // candidate threshold on the raw logit: x / T + G_max >= best - slack
            float x_thr = (fmaxf(bound, best) - kGumbelMax - kCandidateSlack) * p.temperature;
            for (int j0 = warp * 32; j0 < nvec; j0 += kK1Warps * 32) {
                const int j = j0 + lane;
                bool cand[GPV];
#pragma unroll
                for (int g = 0; g < GPV; ++g) cand[g] = false;
                float x[VN], e[VN];  // logits and e = exp((x - m) / T) against the lane's running max m
                if (j < nvec) {
                    Vec<DT>::load(slot + (size_t)j * 16, x);
                    const int base = j * VN;
                    if (base + VN > n_el) {
#pragma unroll
                        for (int i = 0; i < VN; ++i)
                            if (base + i >= n_el) x[i] = -INFINITY;
                    }
                    float gmax[GPV];
#pragma unroll
                    for (int g = 0; g < GPV; ++g)
                        gmax[g] = fmaxf(fmaxf(x[4 * g], x[4 * g + 1]), fmaxf(x[4 * g + 2], x[4 * g + 3]));
                    float vmax = gmax[0];
#pragma unroll
                    for (int g = 1; g < GPV; ++g) vmax = fmaxf(vmax, gmax[g]);
                    // online softmax state
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
                        st.idx = e_lo + base + i0;
                    }
                    if (vmax == st.m) {
                        if (vmax == -INFINITY) {
#pragma unroll
                            for (int i = 0; i < VN; ++i) {
                                bad |= (x[i] != x[i]);
                                e[i] = 0.f;
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < VN; ++i) {
                                if (x[i] == st.m) {
                                    st.c += 1.f;
                                    e[i] = 1.f;
                                } else {
                                    // -inf entries (masked tail, or -inf logits) contribute e = 0;
                                    // the clamp keeps e * d at 0 instead of 0 * -inf
                                    const float d = max_nan((x[i] - st.m) * k2, kMinExponent);
                                    e[i] = ex2(d);
                                    st.r += e[i];
                                    st.t = fmaf(e[i], d, st.t);
                                }
                            }
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < VN; ++i) {
                            const float d = max_nan((x[i] - st.m) * k2, kMinExponent);
                            e[i] = ex2(d);
                            st.r += e[i];
                            st.t = fmaf(e[i], d, st.t);
                        }
                    }
                    if (do_sample) {
#pragma unroll
                        for (int g = 0; g < GPV; ++g) cand[g] = gmax[g] >= x_thr;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < VN; ++i) {
                        x[i] = -INFINITY;
                        e[i] = 0.f;
                    }
                }
                if (!do_sample) continue;
                const float bnd = fmaxf(bound, best);
                bool any = false;
#pragma unroll
                for (int g = 0; g < GPV; ++g) any |= cand[g];
                const unsigned dense_mk = __ballot_sync(0xffffffffu, any);
                if (bnd > -INFINITY && __popc(dense_mk) >= 16) {
                    // Dense: most lanes hold candidates, so every lane draws its own groups' noise.
                    // exp(y - bnd) = e * exp(m / T - bnd) reuses the softmax term; entries with
                    // u <= 1 - 2 exp(y - bnd) cannot beat the bound (see eval_group).
                    const float cb = ex2((st.m * invT - bnd) * kLog2e);
                    const float nscale = -2.f * cb;
#pragma unroll
                    for (int g = 0; g < GPV; ++g) {
                        if (!cand[g]) continue;
                        const int e0 = e_lo + (j * GPV + g) * 4;
                        const dg::u4 w = dg::philox10((uint32_t)e0 >> 2, (uint32_t)pos, step, c3, k0, k1);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float u = dg::uniform_from_word(word_of(w, i));
                            if (!(u > fmaf(nscale, e[4 * g + i], 1.f))) continue;
                            if (e0 + i >= V) continue;
                            const float score = x[4 * g + i] * invT + (-logf(-logf(u)));
                            if (better(score, e0 + i, best, bidx)) {
                                best = score;
                                bidx = e0 + i;
                            }
                        }
                    }
                    warp_best(best, bidx);
                    x_thr = (fmaxf(bound, best) - kGumbelMax - kCandidateSlack) * p.temperature;
                    continue;
                }
                if (!do_sample) continue;
                // queue the candidate groups (ballot-compacted) and draw 32 at a time
#pragma unroll
                for (int g = 0; g < GPV; ++g) {
                    const unsigned mk = __ballot_sync(0xffffffffu, cand[g]);
                    if (cand[g]) {
                        const int at = qn + __popc(mk & lt);
                        uint32_t wv[4];
                        group_words<DT>(x, g, wv);
                        q_e0[at] = e_lo + (j * GPV + g) * 4;
#pragma unroll
                        for (int i = 0; i < QW; ++i) q_x[at][i] = wv[i];
                    }
                    qn += __popc(mk);
                }
                __syncwarp();
                while (qn >= 32) {  // at most 31 + 32 * GPV < 96 entries are queued
                    {
                        float xg[4];
                        words_group<DT>(q_x[lane], xg);
                        eval_group(xg, q_e0[lane], V, invT, (uint32_t)pos, step, c3, k0, k1, bound, best, bidx);
                    }
                    __syncwarp();
                    const int rest = qn - 32;  // move the unprocessed tail to the front
                    for (int r0 = 0; r0 < rest; r0 += 32) {
                        const int r = r0 + lane;
                        int e0v = 0;
                        uint32_t wv[4] = {0u, 0u, 0u, 0u};
                        if (r < rest) {
                            e0v = q_e0[32 + r];
#pragma unroll
                            for (int i = 0; i < QW; ++i) wv[i] = q_x[32 + r][i];
                        }
                        __syncwarp();
                        if (r < rest) {
                            q_e0[r] = e0v;
#pragma unroll
                            for (int i = 0; i < QW; ++i) q_x[r][i] = wv[i];
                        }
                        __syncwarp();
                    }
                    qn = rest;
                    warp_best(best, bidx);
                    x_thr = (fmaxf(bound, best) - kGumbelMax - kCandidateSlack) * p.temperature;
                }
            }
            if (do_sample) {
                // share the best score with the other warps, take theirs
                if (lane == 0 && best > -INFINITY) atomicMax(&sh.best_key, float_key(best));
                __syncwarp();
                bound = fmaxf(bound, key_float(*(volatile unsigned*)&sh.best_key));
            }
            __syncwarp();
            if (lane == 0) dg::mbar_arrive(&sh.empty[sl]);
        }
        if (do_sample && lane < qn) {  // the last (fewer than 32) queued groups
            float xg[4];
            words_group<DT>(q_x[lane], xg);
            eval_group(xg, q_e0[lane], V, invT, (uint32_t)pos, step, c3, k0, k1, bound, best, bidx);
        }
        __syncwarp();
        if (bad) sh.bad = 1;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) st = merge(st, shfl_state(st, o), k2);
        warp_best(best, bidx);
        if (lane == 0) {
            sh.warp_state[warp] = st;
            sh.warp_best[warp] = best;
            sh.warp_bidx[warp] = bidx;
        }
    }
    __syncthreads();
    if (warp == 0) {
        // the sample: the best of the warps' own winners
        float b = -INFINITY;
        int bi = 0x7fffffff;
        if (lane < kK1Warps) {
            b = sh.warp_best[lane];
            bi = sh.warp_bidx[lane];
        }
        warp_best(b, bi);
        if (lane == 0) {
            RowState rs = sh.warp_state[0];
            for (int w = 1; w < kK1Warps; ++w) rs = merge(rs, sh.warp_state[w], k2);
            const bool empty = rs.m == -INFINITY;
            const bool row_bad = sh.bad || rs.m == INFINITY || !isfinite(rs.r) || !isfinite(rs.t);
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
            if (sh.timeout) dg::raise_status(status, DG_DEV_TIMEOUT);
        }
    }
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

// Rows stream through the ring, so any V works up to 2^31 bytes per row.
bool k1_supported(dg_dtype dt, int64_t V) {
    const int64_t es = dt == DG_BF16 ? 2 : 4;
    return V * es < (1LL << 31);
}

template <int DT>
size_t k1_smem_bytes() { return ((sizeof(K1Shared<DT>) + 127) / 128) * 128 + (size_t)kSlots * kPieceBytes; }

template <int DT>
dg_status launch_k1(const void* logits, int64_t ld, int64_t n, int32_t L, int64_t V,
                    const dg_canvas_params* params, uint64_t seed, int32_t* argmax, int32_t* sample, float* entropy,
                    float* lse, cudaStream_t stream) {
    auto kern = k1_row_stats<DT>;
    const size_t smem = k1_smem_bytes<DT>();
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return DG_ERR_CUDA;
    const int64_t ld_bytes = ld * (DT == 0 ? 2 : 4);
    kern<<<dim3((unsigned)L, (unsigned)n, 1), kK1Threads, smem, stream>>>(static_cast<const unsigned char*>(logits),
                                                                          ld_bytes, V, L, params, seed, argmax,
                                                                          sample, entropy, lse, dghost::status_word());
    dghost::count_launch();
    return dghost::cuda_status(cudaGetLastError());
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
    if (!k1_supported(dtype, V)) return DG_ERR_UNSUPPORTED;
    cudaStream_t st = (cudaStream_t)stream;
    s = dtype == DG_BF16 ? launch_k1<0>(logits, ld, n_canvas, L, V, params, seed, argmax, sample, entropy, lse, st)
                         : launch_k1<1>(logits, ld, n_canvas, L, V, params, seed, argmax, sample, entropy, lse, st);
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
