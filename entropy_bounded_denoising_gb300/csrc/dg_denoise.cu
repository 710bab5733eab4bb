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
// engine); eight consumer warps read every piece twice from shared memory.  Pass 1 takes
// vector maxima with packed bf16x2 instructions and queues the candidate groups of the
// Gumbel-max search: an entry whose y + G_max (G_max the largest Gumbel value the uniform
// mapping can produce) cannot reach the best score seen so far is skipped without drawing
// its noise.  Pass 2 folds the piece into an online-softmax state (max m, count c of
// entries equal to m, r = sum of the other e^z, t = sum e^z z -- the split keeps
// near-one-hot rows accurate in fp32) against the warp's running max, which changes only
// between passes, so no lane diverges on a new maximum.  Queued groups are drawn a warp's
// worth at a time, with the Philox rounds that do not depend on the entry index computed
// once per row.
// A sample is kept only at an accepted position (a rejected one is renoised in the same
// step), so canvases without DG_SAMPLE_ALL skip the search in the statistics pass; the
// acceptance kernel lists their accepted rows (with each row's maximum, recorded by the
// statistics pass), and a third kernel searches those rows in chunks of up to 16 KB, the
// warps taking groups of consecutive chunks in a grid-stride loop, reading global memory
// directly: few rows are left, so the work is cut finer than a row to keep every SM busy.
// The reduction order depends only on V, so a row's result does not depend on its batch.
#include <cuda_runtime.h>

#include <math.h>

#include <algorithm>
#include <type_traits>

#include "dg_common.cuh"

namespace {

constexpr int kK1Warps = 8;                        // consumer warps
constexpr int kK1Threads = (kK1Warps + 1) * 32;    // + one producer warp
constexpr int kSlots = 4;                          // ring of shared-memory slots
constexpr uint32_t kChunkBytes = 16384;            // deferred sampling: largest bytes of a row per warp item
constexpr uint32_t kChunkMin = 2048;               // and smallest (one batch of loads per lane)
constexpr int kDWarps = 8;                         // deferred sampling: warps per CTA in line
constexpr int kSideWarps = 3;                      // and per CTA beside a GEMM on another stream
constexpr int kDBatch = 4;                         // 16-byte loads in flight per lane
constexpr int64_t kRunsMaxRows = 512;              // deferred sampling: contiguous runs up to this many rows
constexpr uint32_t kPieceBytes = 16384;            // bytes per slot
constexpr int kVecPerLane = (int)(kPieceBytes / 16) / (kK1Warps * 32);  // 16-byte vectors per lane per piece
constexpr int kDrawPerLane = 1;                    // queued groups drawn per lane per round
constexpr int kDraw = 32 * kDrawPerLane;           // groups drawn per round
constexpr int kQueue = kDrawPerLane == 1 ? 64 : 96;  // per-warp ring of candidate groups awaiting their draw
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Largest Gumbel value the uniform mapping can produce, -log(-log(1 - 2^-24)) = 16.6355...,
// rounded up; plus a margin for the candidate test.
constexpr float kGumbelMax = 16.64f;
constexpr float kCandidateSlack = 1e-3f;
// Smallest Gumbel value, -log(-log(2^-24)) = -2.81153..., by magnitude, rounded up.
constexpr float kGumbelLow = 2.8117f;
// Exponents (log2 units) below this give 2^d = 0 in fp32 with flush-to-zero.
constexpr float kMinExponent = -256.f;
// bf16 pairs: -inf, and -2^64 (the floor applied to logits before the exponent, so that a
// -inf logit gives e = 0 and e * d = 0 instead of 0 * -inf).
constexpr uint32_t kBf16NegInf2 = 0xFF80FF80u;
constexpr uint32_t kBf16NegFloor2 = 0xDF80DF80u;

static_assert(kVecPerLane * kK1Warps * 32 * 16 == (int)kPieceBytes, "a piece splits evenly over the lanes");

struct RowState {  // online softmax state of a set of entries, z measured in log2 units
    float m;       // reference: the largest raw logit seen by the warp (-inf = empty)
    float c;       // entries equal to m
    float r;       // sum of 2^d over the other entries, d = (x - m) * log2e / T
    float t;       // sum of 2^d * d
    int idx;       // smallest index attaining m
};

// The deferred-sampling workspace (caller memory, carved by dg_denoise_step): the list of
// accepted rows of canvases without DG_SAMPLE_ALL, filled by the acceptance kernel.
struct DeferredWs {
    int32_t* count;  // entries listed
    int2* entry;     // [n * L]: (row, bits of the row's largest raw logit)
    unsigned long long* key;  // [n * L]: best (score, entry) of the row so far, see score_key
    int32_t* done;   // [n * L]: chunks of the row searched so far
    float* row_max;  // [n * L] by row: written by the statistics pass
    int32_t all_deferred;  // 1: every canvas is sampled by the deferred pass (DG_SAMPLE_ALL ignored)
};

// Optional single-pass-read output of the statistics pass: per active position, the
// probabilities of C caller-given tokens under the position's own softmax(logits / T).
struct ChoiceOut {
    const int32_t* choices;  // [rows][C]; a token outside [0, V) gives probability 0
    float* probs;            // [rows][C]; null: nothing gathered
    int32_t C;
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
    // per-warp ring of candidate groups: first entry index and the 4 logits (raw words), so
    // a queued group outlives the ring slot it came from
    int q_e0[kK1Warps][kQueue];
    uint32_t q_x[kK1Warps][kQueue][kQW];
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

// Lane-wise max of two bf16 pairs, NaN-propagating.
DG_DEVINL uint32_t bmax2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Either half of bf16 pair a >= (==) the same half of b.
DG_DEVINL bool bge2_any(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("{\n\t.reg .pred p, q;\n\tsetp.ge.bf16x2 p|q, %1, %2;\n\tor.pred p, p, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(a), "r"(b));
    return r != 0;
}
DG_DEVINL bool beq2_any(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("{\n\t.reg .pred p, q;\n\tsetp.eq.bf16x2 p|q, %1, %2;\n\tor.pred p, p, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(a), "r"(b));
    return r != 0;
}

DG_DEVINL float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
DG_DEVINL float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// The largest bf16 value <= t, in both halves of a pair (a conservative candidate threshold).
DG_DEVINL uint32_t bf16_floor2(float t) {
    const uint32_t b = __float_as_uint(t);
    uint32_t h = b >> 16;                                      // truncation: toward zero
    if ((b & 0xffffu) != 0u && (b & 0x80000000u) != 0u && t == t) h += 1u;  // negative: one step down
    if (t != t) h = 0xFF80u;
    return h | (h << 16);
}

// (lo - m, hi - m) for a bf16 pair, each with the mixed-precision subtract (bf16 operand, fp32
// result): the bf16 value widens exactly and, with m itself a bf16 value, the difference is
// exact in fp32 -- the same result as unpacking first, without the unpacking instructions.
DG_DEVINL void bf16x2_sub_f32(uint32_t w, float m, float& lo, float& hi) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tsub.rn.f32.bf16 %0, l, %3;\n\t"
        "sub.rn.f32.bf16 %1, h, %3;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(w), "f"(m));
}

// Packed fp32 pairs (sm_100 f32x2 arithmetic, round to nearest like the scalar forms).
DG_DEVINL uint64_t f2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
DG_DEVINL float f2_lo(uint64_t v) { return __uint_as_float((uint32_t)v); }
DG_DEVINL float f2_hi(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
DG_DEVINL uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
DG_DEVINL uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
DG_DEVINL uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
DG_DEVINL uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
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

// Index into a warp's candidate ring, for arguments below 2 * kQueue.
DG_DEVINL int queue_slot(int i) { return (kQueue & (kQueue - 1)) == 0 ? (i & (kQueue - 1)) : (i >= kQueue ? i - kQueue : i); }
static_assert(kDraw - 1 + 32 <= kQueue, "a round's worth of groups plus one vector's fit the ring");

template <int DT>
struct Vec {  // 16 bytes of logits: 8 bf16 or 4 fp32 entries
    static constexpr int N = DT == 0 ? 8 : 4;
};

// The 16-byte vector j of a slot as raw words, entries past the row's end (or vectors past
// the piece's end) set to -inf.  FULL: the piece is whole, no checks.
template <int DT, bool FULL>
DG_DEVINL uint4 load_raw(const unsigned char* slot, int j, int nvec, int n_el) {
    constexpr int VN = Vec<DT>::N;
    constexpr uint32_t kNegInf = DT == 0 ? kBf16NegInf2 : 0xFF800000u;
    if (FULL) return *reinterpret_cast<const uint4*>(slot + (size_t)j * 16);
    uint4 w = make_uint4(kNegInf, kNegInf, kNegInf, kNegInf);
    if (j < nvec) {
        w = *reinterpret_cast<const uint4*>(slot + (size_t)j * 16);
        const int valid = n_el - j * VN;
        if (valid < VN) {  // the row's ragged end
            uint32_t a[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < VN; ++i) {
                if (i < valid) continue;
                if (DT == 0)
                    a[i >> 1] = (i & 1) ? ((a[i >> 1] & 0x0000ffffu) | 0xFF800000u) : ((a[i >> 1] & 0xffff0000u) | 0xFF80u);
                else
                    a[i] = 0xFF800000u;
            }
            w = make_uint4(a[0], a[1], a[2], a[3]);
        }
    }
    return w;
}

template <int DT>
DG_DEVINL void unpack(const uint4& w, float (&x)[Vec<DT>::N]) {
    if constexpr (DT == 0) {
        x[0] = bf_lo(w.x); x[1] = bf_hi(w.x); x[2] = bf_lo(w.y); x[3] = bf_hi(w.y);
        x[4] = bf_lo(w.z); x[5] = bf_hi(w.z); x[6] = bf_lo(w.w); x[7] = bf_hi(w.w);
    } else {
        x[0] = __uint_as_float(w.x); x[1] = __uint_as_float(w.y);
        x[2] = __uint_as_float(w.z); x[3] = __uint_as_float(w.w);
    }
}

template <int DT>
DG_DEVINL void words_group(const uint32_t* w, float (&x)[4]) {
    if (DT == 0) {
        x[0] = bf_lo(w[0]); x[1] = bf_hi(w[0]); x[2] = bf_lo(w[1]); x[3] = bf_hi(w[1]);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = __uint_as_float(w[i]);
    }
}

// Gumbel draw for one group of 4 consecutive entries (one Philox block, words w) [e0, e0 + 4)
// with logits x.  Keeps (best, bidx) as the largest score y + g, y = x / T, ties to the
// lower index.  Entries that cannot reach max(bound, best) are not drawn: g > D needs
// u > exp(-e^-D) >= 1 - e^-D, tested (with a factor 2 of slack) first for the whole group
// against its largest uniform and largest logit, then per entry.
DG_DEVINL void eval_words(const float (&x)[4], int e0, const dg::u4& w, int64_t V, float invT, float bound,
                          float& best, int& bidx) {
    {
        const float b = fmaxf(bound, best);
        const float ymax = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])) * invT;
        const float umax = dg::uniform_from_word(max(max(w.x, w.y), max(w.z, w.w)));
        if (!(umax > 1.f - 2.f * ex2((ymax - b) * kLog2e))) return;
    }
#pragma unroll 1
    for (int i = 0; i < 4; ++i) {  // rare (a few groups per row): kept rolled, small code
        if (e0 + i >= V) continue;
        const float y = (i == 0 ? x[0] : i == 1 ? x[1] : i == 2 ? x[2] : x[3]) * invT;
        const float b = fmaxf(bound, best);
        if (!(y >= b - kGumbelMax - kCandidateSlack)) continue;
        const float u = dg::uniform_from_word(word_of(w, i));
        const float eb = 2.f * ex2(-(b - y) * kLog2e);
        if (!(u > 1.f - eb)) continue;
        const float score = y + (-logf(-logf(u)));
        if (better(score, e0 + i, best, bidx)) {
            best = score;
            bidx = e0 + i;
        }
    }
}

// Queued groups of one warp: kDraw at a time, kDrawPerLane per lane (independent Philox
// chains), or the fewer left at the end of the row.  All 32 lanes call it (warp-uniform n).
template <int DT, int QW>
DG_DEVINL void draw_queued(const int* q_e0, const uint32_t (*q_x)[QW], int qh, int n, int lane, int64_t V,
                           float invT, const dg::PhiloxPre& pre, float bound, float& best, int& bidx) {
    float xs[kDrawPerLane][4];
    int es[kDrawPerLane];
#pragma unroll
    for (int r = 0; r < kDrawPerLane; ++r) {
        const int at = queue_slot(qh + 32 * r + lane);
        words_group<DT>(q_x[at], xs[r]);
        es[r] = q_e0[at];
    }
    __syncwarp();  // read before later groups reuse these entries
    dg::u4 w[kDrawPerLane];
#pragma unroll
    for (int r = 0; r < kDrawPerLane; ++r) w[r] = dg::philox10_c0((uint32_t)es[r] >> 2, pre);
#pragma unroll
    for (int r = 0; r < kDrawPerLane; ++r)
        if (32 * r + lane < n) eval_words(xs[r], es[r], w[r], V, invT, bound, best, bidx);
}

// ------------------------------------------------------------------------------------
// K1: per-position statistics and Gumbel-max sample.  grid (L, n), one CTA per position.
// Each consumer warp takes kVecPerLane 16-byte vectors per lane of every piece, in two
// passes over shared memory: (1) vector maxima, candidate groups into the warp's queue;
// (2) the exponential sums against the warp's running max, which only grows between
// pieces (a warp-uniform branch), so lanes do not diverge on new maxima.
// ------------------------------------------------------------------------------------
// ws (may be null): the deferred-sampling workspace; its list count is cleared here (before
// any CTA returns) and each row's largest raw logit recorded (NaN for a NaN / inf / empty row).
template <int DT>
__global__ void __launch_bounds__(kK1Threads, 3) k1_row_stats(
    const unsigned char* __restrict__ logits, int64_t ld_bytes, int64_t V, int32_t L,
    const dg_canvas_params* __restrict__ params, uint64_t seed, int32_t* __restrict__ argmax_out,
    int32_t* __restrict__ sample_out, float* __restrict__ entropy_out, float* __restrict__ lse_out,
    DeferredWs ws, ChoiceOut co, unsigned* status) {
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

    dg::pdl_wait();
    dg::pdl_release();
    if (ws.count && pos == 0 && canvas == 0 && tid == 0) *ws.count = 0;
    const dg_canvas_params p = params[canvas];
    if (!(p.flags & DG_ACTIVE)) return;
    if (!(p.temperature > 0.f) || !isfinite(p.temperature)) {
        if (tid == 0 && pos == 0) dg::raise_status(status, DG_DEV_BAD_PARAM);
        return;
    }
    const int64_t row = canvas * L + pos;
    const unsigned char* src = logits + row * ld_bytes;
    const bool do_sample = (p.flags & DG_SAMPLE_ALL) && !(p.flags & DG_READ_ONLY);
    const float invT = 1.0f / p.temperature;
    const float k2 = kLog2e * invT;
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
        float best = -INFINITY;    // this lane's best score and its entry
        int bidx = 0x7fffffff;
        float bound = -INFINITY;   // best score known anywhere in the CTA
        const dg::PhiloxPre pre = dg::philox_pre((uint32_t)pos, (uint32_t)p.step,
                                                 dg::ctr_word3(seed, dg::kStreamGumbel), (uint32_t)seed, p.request_id);
        int* q_e0 = sh.q_e0[warp];
        uint32_t(*q_x)[QW] = sh.q_x[warp];
        int qh = 0, qn = 0;  // warp-uniform queue head and length, kept across pieces
        const unsigned lt = (1u << lane) - 1u;
        for (int q = 0; q < npieces; ++q) {
            const int sl = q % kSlots;
            if (!__all_sync(0xffffffffu, dg::mbar_wait(&sh.full[sl], (uint32_t)(q / kSlots) & 1u))) {
                sh.timeout = 1;
                break;
            }
            const unsigned char* slot = ring + (size_t)sl * kPieceBytes;
            const int e_lo = q * kPieceElems;
            const int n_el = (int)min((int64_t)kPieceElems, V - e_lo);
            const int nvec = (n_el + VN - 1) / VN;

            // One piece in two passes; FULL: every vector of the piece is whole (all but the
            // row's last piece), so the bounds checks drop out; SAMPLE: the Gumbel-max search
            // runs (not for read-only canvases).
            auto piece = [&](auto full_tag, auto sample_tag) {
                constexpr bool FULL = decltype(full_tag)::value;
                constexpr bool SAMPLE = decltype(sample_tag)::value;
                // ---- pass 1: vector maxima, then the warp's max; a larger one rescales every
                // lane's state (warp-uniform, so lanes never diverge on a new maximum)
                uint32_t lm2 = kBf16NegInf2;  // lane max as a bf16 pair (max of even, odd entries)
                float lane_max = -INFINITY;
#pragma unroll
                for (int v = 0; v < kVecPerLane; ++v) {
                    const int j = (v * kK1Warps + warp) * 32 + lane;
                    const uint4 w = load_raw<DT, FULL>(slot, j, nvec, n_el);
                    if constexpr (DT == 0) {
                        lm2 = bmax2(lm2, bmax2(bmax2(w.x, w.y), bmax2(w.z, w.w)));
                    } else {
                        const float vmax = max_nan(max_nan(__uint_as_float(w.x), __uint_as_float(w.y)),
                                                   max_nan(__uint_as_float(w.z), __uint_as_float(w.w)));
                        lane_max = max_nan(lane_max, vmax);
                    }
                }
                if (DT == 0) lane_max = max_nan(bf_lo(lm2), bf_hi(lm2));
                float wmax = lane_max;
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) wmax = max_nan(wmax, __shfl_xor_sync(0xffffffffu, wmax, o));
                if (wmax != wmax) {
                    bad = true;
                } else if (wmax > st.m) {
                    if (st.m > -INFINITY) {
                        const float d = (st.m - wmax) * k2, al = ex2(d), s = st.c + st.r;
                        st.t = al * (st.t + d * s);
                        st.r = al * s;
                    }
                    st.c = 0.f;
                    st.m = wmax;
                    st.idx = 0x7fffffff;
                }
                if (!(st.m > -INFINITY && st.m < INFINITY)) return;  // nothing to add while m = -inf

                // ---- pass 2: candidate groups and exponential sums.  Every score is at least
                // its y plus the smallest Gumbel value, so m / T - kGumbelLow bounds the winner's
                // score from below before any noise is drawn.  x - m is exact for bf16 entries,
                // so d carries one rounding whatever the size of m / T.
                const float ym = st.m * invT;
                bound = fmaxf(bound, ym - kGumbelLow - fabsf(ym) * 2.4e-7f);
                const float x_thr = (fmaxf(bound, best) - kGumbelMax - kCandidateSlack) * p.temperature;
                const uint32_t thr2 = DT == 0 ? bf16_floor2(x_thr) : 0u;
                const uint32_t m2 = DT == 0 ? (__float_as_uint(st.m) >> 16) * 0x10001u : 0u;
                (void)thr2;
                (void)m2;
                const uint64_t mm = f2(st.m, st.m), kk = f2(k2, k2);
                uint64_t racc[2] = {0ull, 0ull}, tacc[2] = {0ull, 0ull};  // pairs of partial sums
                // TIE: the vector may hold entries equal to the running max (counted in c).  Only a
                // lane whose own maximum over this piece equals it can hold one, so a piece without
                // such a lane (a warp vote) skips the per-vector test.
                auto vec2 = [&](int v, auto tie_tag) {
                    constexpr bool TIE = decltype(tie_tag)::value;
                    const int j = (v * kK1Warps + warp) * 32 + lane;
                    const bool in = FULL || j < nvec;
                    const uint4 w = load_raw<DT, FULL>(slot, j, nvec, n_el);
                    bool cand[GPV], tie = false;
                    if constexpr (DT == 0) {
                        const uint32_t g0 = bmax2(w.x, w.y), g1 = bmax2(w.z, w.w);
                        cand[0] = SAMPLE && in && bge2_any(g0, thr2);
                        cand[GPV - 1] = SAMPLE && in && bge2_any(g1, thr2);
                        if (TIE) tie = beq2_any(bmax2(g0, g1), m2);
                    } else {
                        const float vmax = max_nan(max_nan(__uint_as_float(w.x), __uint_as_float(w.y)),
                                                   max_nan(__uint_as_float(w.z), __uint_as_float(w.w)));
                        cand[0] = SAMPLE && in && vmax >= x_thr;
                        if (TIE) tie = vmax == st.m;
                    }
                    if (in) {
                        float x[VN];
                        if (tie) {
                            // the vector holds the max: count its copies, the rest as usual
                            unpack<DT>(w, x);
        #pragma unroll
                            for (int i = 0; i < VN; ++i) {
                                if (x[i] == st.m) {
                                    st.c += 1.f;
                                    st.idx = min(st.idx, e_lo + j * VN + i);
                                } else {
                                    const float d = max_nan((x[i] - st.m) * k2, kMinExponent);
                                    const float e = ex2(d);
                                    st.r += e;
                                    st.t = fmaf(e, d, st.t);
                                }
                            }
                        } else if constexpr (DT == 0) {
                            // entries floored at -2^64 (a -inf logit gives e = 0, e * d = 0), two per op
                            const uint32_t fw[4] = {bmax2(w.x, kBf16NegFloor2), bmax2(w.y, kBf16NegFloor2),
                                                    bmax2(w.z, kBf16NegFloor2), bmax2(w.w, kBf16NegFloor2)};
        #pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                float dl, dh;
                                bf16x2_sub_f32(fw[k], st.m, dl, dh);
                                const uint64_t d2 = f2_mul(f2(dl, dh), kk);
                                const uint64_t e2 = f2(ex2(f2_lo(d2)), ex2(f2_hi(d2)));
                                racc[k & 1] = f2_add(racc[k & 1], e2);
                                tacc[k & 1] = f2_fma(e2, d2, tacc[k & 1]);
                            }
                        } else {
                            unpack<DT>(w, x);
        #pragma unroll
                            for (int i = 0; i < VN; ++i) {
                                const float d = max_nan((x[i] - st.m) * k2, kMinExponent);
                                const float e = ex2(d);
                                st.r += e;
                                st.t = fmaf(e, d, st.t);
                            }
                        }
                    }
                    if (!SAMPLE) return;
                    bool any = false;
        #pragma unroll
                    for (int g = 0; g < GPV; ++g) any |= cand[g];
                    if (__ballot_sync(0xffffffffu, any) == 0u) return;
        #pragma unroll
                    for (int g = 0; g < GPV; ++g) {
                        const unsigned mk = __ballot_sync(0xffffffffu, cand[g]);
                        if (cand[g]) {
                            const int at = queue_slot(qh + qn + __popc(mk & lt));
                            q_e0[at] = e_lo + (j * GPV + g) * 4;
                            if (DT == 0) {
                                q_x[at][0] = g == 0 ? w.x : w.z;
                                q_x[at][1] = g == 0 ? w.y : w.w;
                            } else {
                                q_x[at][0] = w.x;
                                q_x[at][1] = w.y;
                                if (QW == 4) {
                                    q_x[at][QW - 2] = w.z;
                                    q_x[at][QW - 1] = w.w;
                                }
                            }
                        }
                        qn += __popc(mk);
                        __syncwarp();
                        if (qn >= kDraw) {  // at most kDraw - 1 + 32 <= kQueue groups are queued
                            draw_queued<DT, QW>(q_e0, q_x, qh, kDraw, lane, V, invT, pre, bound, best, bidx);
                            qh = queue_slot(qh + kDraw);
                            qn -= kDraw;
                        }
                    }
                };
                if constexpr (SAMPLE) {
#pragma unroll 1
                    for (int v = 0; v < kVecPerLane; ++v) vec2(v, std::true_type{});  // rolled: one copy of the draw code
                } else if (FULL && !__any_sync(0xffffffffu, lane_max == st.m)) {
#pragma unroll
                    for (int v = 0; v < kVecPerLane; ++v) vec2(v, std::false_type{});
                } else {
#pragma unroll
                    for (int v = 0; v < kVecPerLane; ++v) vec2(v, std::true_type{});
                }
                if (DT == 0) {
                    st.r += (f2_lo(racc[0]) + f2_hi(racc[0])) + (f2_lo(racc[1]) + f2_hi(racc[1]));
                    st.t += (f2_lo(tacc[0]) + f2_hi(tacc[0])) + (f2_lo(tacc[1]) + f2_hi(tacc[1]));
                }
            };
            if (do_sample) {
                if (n_el == kPieceElems) piece(std::true_type{}, std::true_type{});
                else piece(std::false_type{}, std::true_type{});
            } else {
                if (n_el == kPieceElems) piece(std::true_type{}, std::false_type{});
                else piece(std::false_type{}, std::false_type{});
            }

            if (do_sample) {
                // share the best score with the other warps, take theirs
                warp_best(best, bidx);
                const float mine = fmaxf(best, bound);
                if (lane == 0 && mine > -INFINITY) atomicMax(&sh.best_key, float_key(mine));
                __syncwarp();
                bound = fmaxf(bound, key_float(*(volatile unsigned*)&sh.best_key));
            }
            __syncwarp();
            if (lane == 0) dg::mbar_arrive(&sh.empty[sl]);
        }
        if (do_sample && qn > 0) draw_queued<DT, QW>(q_e0, q_x, qh, qn, lane, V, invT, pre, bound, best, bidx);
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
        float lse = 0.f;
        if (lane == 0) {
            RowState rs = sh.warp_state[0];
            for (int w = 1; w < kK1Warps; ++w) rs = merge(rs, sh.warp_state[w], k2);
            const bool empty = rs.m == -INFINITY;
            const bool row_bad = sh.bad || rs.m == INFINITY || !isfinite(rs.r) || !isfinite(rs.t);
            // H = log(c + r) - t ln2 / (c + r), with log1p where a single entry holds the max
            const float s = rs.c + rs.r;
            const float lns = (rs.c == 1.f) ? log1pf(rs.r) : logf(rs.c) + log1pf(rs.r / rs.c);
            const float H = lns - rs.t * kLn2 / s;
            lse = rs.m * invT + lns;
            entropy_out[row] = H;
            lse_out[row] = lse;
            argmax_out[row] = empty ? 0 : rs.idx;
            sample_out[row] = (do_sample && !empty && !row_bad) ? bi : -1;
            if (ws.row_max) ws.row_max[row] = (empty || row_bad) ? __int_as_float(0x7fc00000) : rs.m;
            if (row_bad) dg::raise_status(status, DG_DEV_NAN_INF_ROW);
            if (empty) dg::raise_status(status, DG_DEV_EMPTY_ROW);
            if (sh.timeout) dg::raise_status(status, DG_DEV_TIMEOUT);
        }
        if (co.probs) {
            // choice probabilities from the lse just formed; the chosen logits come from the
            // row that was streamed a moment ago (L2)
            lse = __shfl_sync(0xffffffffu, lse, 0);
            const int32_t* ch = co.choices + row * co.C;
            float* pr = co.probs + row * co.C;
            for (int k = lane; k < co.C; k += 32) {
                const int32_t tok = ch[k];
                float out = 0.f;
                if (tok >= 0 && (int64_t)tok < V) {
                    const float x = DT == 0 ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(src)[tok] << 16)
                                            : reinterpret_cast<const float*>(src)[tok];
                    out = expf(x * invT - lse);
                }
                pr[k] = out;
            }
        }
    }
}

// ------------------------------------------------------------------------------------
// Deferred sampling: the Gumbel-max samples of the listed accepted rows.  Work items are
// (list entry, chunk of its row), taken in groups of consecutive items by the warps in a
// grid-stride loop (a warp streams each row's part of its group as one segment and publishes
// once per segment); chunks are 16 KB,
// or shorter (down to 2 KB) when the listed rows are too few to give every warp two; a lane
// loads kDBatch 16-byte vectors at a time straight from global memory and draws the noise
// only for 4-entry groups whose largest y + G_max reaches the bound m / T - kGumbelLow (m
// the row's largest logit) or the warp's best so far.  A segment's winner joins the row's
// 64-bit key by atomicMax (order-independent, so the result is deterministic) and its chunks
// are added to the row's count; the warp that brings the count to the row's chunks writes
// its sample and token.
// ------------------------------------------------------------------------------------
// Order-preserving key of (score, entry): larger score first, then the smaller entry.
DG_DEVINL unsigned long long score_key(float score, int idx) {
    return ((unsigned long long)float_key(score) << 32) | (unsigned long long)(0xffffffffu - (uint32_t)idx);
}

// kRuns: each warp takes one contiguous run of the items (for short lists, where a warp
// gets at most a few chunks: a second chunk of the same row then costs no second
// publication); else one chunk per step of a grid-stride loop, so that the warps read one
// compact window of the list at a time (measured: contiguous runs are slower on long lists).
// kW warps per CTA: 8 in line (3 CTAs per SM), 3 beside a GEMM on another stream (96 threads
// x 80 registers fit next to a P.E CTA's 448 x 128 in an SM's 64 K registers).
template <int DT, bool kRuns, int kW>
__global__ void __launch_bounds__(kW * 32, kW == kDWarps ? 3 : 8) k1_sample_listed(
    const unsigned char* __restrict__ logits, int64_t ld_bytes, int64_t V, int32_t L,
    const dg_canvas_params* __restrict__ params, uint64_t seed, DeferredWs ws, int32_t* __restrict__ sample_out,
    int32_t* __restrict__ canvas_out, int64_t rows) {
    constexpr int VN = Vec<DT>::N;
    constexpr int ES = DT == 0 ? 2 : 4;
    constexpr int GPV = VN / 4;
    static_assert(kChunkMin % (32 * kDBatch * 16) == 0 && kChunkBytes % kChunkMin == 0, "whole batches per chunk");
    const int lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * kW + (threadIdx.x >> 5);
    const int64_t nw = (int64_t)gridDim.x * kW;
    dg::pdl_wait();
    dg::pdl_release();
    const int count = *ws.count;
    // chunk size: every warp computes the same one from the list length (in float: the size
    // only cuts the work, the result does not depend on it; 64-bit divisions are long
    // emulated sequences)
    const int64_t row_bytes = V * ES;  // < 2^31
    const float want = (float)count * (float)row_bytes / (float)(2 * nw);
    const uint32_t chunk_bytes =
        want >= (float)kChunkBytes ? kChunkBytes
                                   : max(kChunkMin, ((uint32_t)want + kChunkMin - 1) / kChunkMin * kChunkMin);
    const int kChunkElems = (int)(chunk_bytes / ES);
    const int cpr = (int)(((uint32_t)row_bytes + chunk_bytes - 1) / chunk_bytes);  // chunks per row
    const int64_t items = (int64_t)count * cpr;
    const bool items32 = items <= 0xffffffffLL;  // item indices split in 32-bit arithmetic
    // One row segment: chunks [c_lo, c_hi) of list entry w, searched and published (the
    // winner into the row's key, the chunks into its count; the warp that completes the count
    // writes the sample and token).
    auto segment = [&](int w, int c_lo, int c_hi) {
        const int2 e = ws.entry[w];
        const int64_t row = e.x;
        const bool in_range = (uint64_t)row < (uint64_t)rows;  // entries come from K2; checked anyway
        const float m = __int_as_float(e.y);
        const int64_t canvas = in_range ? (int64_t)((uint32_t)row / (uint32_t)L) : 0;  // row < n L < 2^26
        const dg_canvas_params p = params[canvas];
        const bool ok = in_range && isfinite(m);  // else a NaN / inf / empty row (flagged by the statistics pass)
        float best = -INFINITY;
        int bidx = 0x7fffffff;
        if (ok) {
            const int pos = (int)(row - canvas * L);
            const float invT = 1.0f / p.temperature;
            const float ym = m * invT;
            const float bound = ym - kGumbelLow - fabsf(ym) * 2.4e-7f;
            const dg::PhiloxPre pre = dg::philox_pre((uint32_t)pos, (uint32_t)p.step,
                                                     dg::ctr_word3(seed, dg::kStreamGumbel), (uint32_t)seed,
                                                     p.request_id);
            const int e_lo = c_lo * kChunkElems;
            const uint4* src = reinterpret_cast<const uint4*>(logits + row * ld_bytes + (int64_t)e_lo * ES);
            const int n_el = (int)min((int64_t)(c_hi - c_lo) * kChunkElems, V - e_lo);
            const int nvec = (n_el + VN - 1) / VN;
            float x_thr = (bound - kGumbelMax - kCandidateSlack) * p.temperature;
            uint32_t thr2 = DT == 0 ? bf16_floor2(x_thr) : 0u;
            // two register batches: the next one is loading while this one is tested
            uint4 cur[kDBatch], nxt[kDBatch];
            auto load = [&](uint4 (&buf)[kDBatch], int b0) {
#pragma unroll
                for (int k = 0; k < kDBatch; ++k) {
                    const int j = b0 + k * 32 + lane;
                    buf[k] = j < nvec ? __ldcs(src + j) : make_uint4(0, 0, 0, 0);
                }
            };
            load(cur, 0);
#pragma unroll 1
            for (int b0 = 0; b0 < nvec; b0 += 32 * kDBatch) {
                if (b0 + 32 * kDBatch < nvec) load(nxt, b0 + 32 * kDBatch);
                const float best0 = best;
#pragma unroll
                for (int k = 0; k < kDBatch; ++k) {
                    const int j = b0 + k * 32 + lane;
                    if (j >= nvec) continue;
                    const uint4 v = cur[k];
                    const int valid = n_el - j * VN;  // entries of this vector inside the segment
                    bool cand[GPV];
                    if (DT == 0 && valid >= VN) {
                        // whole vector: packed test of each 4-entry group's max
                        cand[0] = bge2_any(bmax2(v.x, v.y), thr2);
                        cand[GPV - 1] = bge2_any(bmax2(v.z, v.w), thr2);
                    } else {
                        float x[VN];
                        unpack<DT>(v, x);
#pragma unroll
                        for (int i = 0; i < VN; ++i)
                            if (i >= valid) x[i] = -INFINITY;
#pragma unroll
                        for (int g = 0; g < GPV; ++g)
                            cand[g] = fmaxf(fmaxf(x[4 * g], x[4 * g + 1]), fmaxf(x[4 * g + 2], x[4 * g + 3])) >= x_thr;
                    }
#pragma unroll
                    for (int g = 0; g < GPV; ++g) {
                        if (!cand[g]) continue;  // rare: a candidate group is drawn where found
                        float x[VN];
                        unpack<DT>(v, x);
#pragma unroll
                        for (int i = 0; i < VN; ++i)
                            if (i >= valid) x[i] = -INFINITY;
                        const int e0 = e_lo + (j * GPV + g) * 4;
                        const float xg[4] = {x[4 * g], x[4 * g + 1], x[4 * g + 2], x[4 * g + 3]};
                        const dg::u4 r = dg::philox10_c0((uint32_t)e0 >> 2, pre);
                        eval_words(xg, e0, r, V, invT, bound, best, bidx);
                    }
                }
                // a lane's new best tightens every lane's threshold for the next batch
                if (__any_sync(0xffffffffu, best != best0)) {
                    warp_best(best, bidx);
                    x_thr = (fmaxf(bound, best) - kGumbelMax - kCandidateSlack) * p.temperature;
                    thr2 = DT == 0 ? bf16_floor2(x_thr) : 0u;
                }
#pragma unroll
                for (int k = 0; k < kDBatch; ++k) cur[k] = nxt[k];
            }
            warp_best(best, bidx);
        }
        if (lane == 0) {
            if (ok && best > -INFINITY) atomicMax(ws.key + w, score_key(best, bidx));
            __threadfence();
            const int nc = c_hi - c_lo;
            if (atomicAdd(ws.done + w, nc) == cpr - nc && in_range) {
                // every chunk of the row is in: its winner is the position's sample and token
                __threadfence();
                const unsigned long long k = atomicMax(ws.key + w, 0ull);
                const int32_t tok = (ok && k != 0ull) ? (int32_t)(0xffffffffu - (uint32_t)(k & 0xffffffffull)) : -1;
                sample_out[row] = tok;
                canvas_out[row] = tok;
            }
        }
        __syncwarp();
    };
    auto row_of = [&](int64_t it) {
        return items32 ? (int)((uint32_t)it / (uint32_t)cpr) : (int)(it / cpr);
    };
    if constexpr (!kRuns) {
        for (int64_t it = gw; it < items; it += nw) {
            const int w = row_of(it);
            const int c = (int)(it - (int64_t)w * cpr);
            segment(w, c, c + 1);
        }
    } else {
        const int64_t per = (items + nw - 1) / nw;
        for (int64_t it = gw * per, it1 = min(items, gw * per + per); it < it1;) {
            const int w = row_of(it);
            const int c_lo = (int)(it - (int64_t)w * cpr);
            const int c_hi = (int)min((int64_t)cpr, (int64_t)c_lo + (it1 - it));
            it += c_hi - c_lo;
            segment(w, c_lo, c_hi);
        }
    }
}

// ------------------------------------------------------------------------------------
// K2: acceptance, renoise and convergence for one canvas per CTA (blockDim = 32 * ceil(L/32)).
// ------------------------------------------------------------------------------------
// kMaxT: 256 (up to 256 positions; 32 registers, so that the CTA fits beside a GEMM CTA on
// another stream) or 1024.  late_release: let the next launch on the stream start only when
// this grid completes (so that a sampler launched after it cannot take an SM that a GEMM on
// another stream is about to need).
template <int kMaxT>
__global__ void __launch_bounds__(kMaxT, kMaxT <= 256 ? 8 : 1) k2_accept(
    const float* __restrict__ entropy, const int32_t* __restrict__ sample, const int32_t* __restrict__ argmax,
    int32_t L, int64_t V, const dg_canvas_params* __restrict__ params, uint64_t seed, int32_t* __restrict__ canvas,
    int32_t* __restrict__ prev_argmax, int32_t* __restrict__ stable_count, uint8_t* __restrict__ accept_mask,
    uint8_t* __restrict__ converged, float* __restrict__ mean_entropy, int32_t* __restrict__ n_accept,
    DeferredWs ws, int late_release, unsigned* status) {
    __shared__ __align__(16) float sH[kMaxT];
    __shared__ double sSorted[kMaxT];
    __shared__ double sWarp[32];
    __shared__ int sCut;
    __shared__ int sBase;

    const int64_t c = blockIdx.x;
    const int i = threadIdx.x, lane = i & 31, warp = i >> 5, nwarps = blockDim.x >> 5;
    dg::pdl_wait();
    if (!late_release) dg::pdl_release();
    const bool valid = i < L;
    const int64_t q = c * L + i;
    // the per-position loads (and the canvas's stable count) go out with the parameter load:
    // in range whatever the parameters say, unused for an inactive canvas
    const float H0 = valid ? entropy[q] : 0.f;
    const int32_t am = valid ? argmax[q] : 0;
    const int32_t pam = valid ? prev_argmax[q] : 0;
    const int32_t st0 = i == 0 ? stable_count[c] : 0;
    const dg_canvas_params p = params[c];
    if (!(p.flags & DG_ACTIVE)) return;
    if (!dg::canvas_params_ok(p, L)) {
        if (i == 0) dg::raise_status(status, DG_DEV_BAD_PARAM);
        return;
    }
    const bool read_only = (p.flags & DG_READ_ONLY) != 0;
    // ws.count null (the acceptance hook): no deferred sampling.  Else accepted positions of
    // a canvas without DG_SAMPLE_ALL are listed for the deferred sampling pass, which writes
    // their sample and token
    const bool deferred = ws.count && (ws.all_deferred || !(p.flags & DG_SAMPLE_ALL));
    // a NaN entropy (a row flagged by the statistics pass) ranks after every number, so the
    // ranks stay a permutation and every reserved slot of the sampler's list is written
    const float H = (H0 == H0) ? H0 : INFINITY;
    const int L4 = (L + 3) & ~3;  // <= blockDim.x
    // +inf pads the entropies to whole quads; a pad never ranks before a position (its index
    // is larger and no entropy exceeds +inf)
    if (valid) sH[i] = H;
    else if (i < L4) sH[i] = INFINITY;
    if (i == 0) sCut = L;
    __syncthreads();

    // rank in (entropy, position) order, four entropies per shared-memory read
    int rk = 0;
    if (valid) {
        const float4* h4 = reinterpret_cast<const float4*>(sH);
#pragma unroll 4
        for (int j = 0; j < L4; j += 4) {
            const float4 hv = h4[j >> 2];
            rk += (hv.x < H) || (hv.x == H && j < i);
            rk += (hv.y < H) || (hv.y == H && j + 1 < i);
            rk += (hv.z < H) || (hv.z == H && j + 2 < i);
            rk += (hv.w < H) || (hv.w == H && j + 3 < i);
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

    if (i == 0 && deferred && nacc > 0) sBase = atomicAdd(ws.count, nacc);
    const bool same = __syncthreads_and(!valid || am == pam) != 0;
    if (valid) {
        const bool acc = rk < nacc;
        if (deferred && acc) {  // accepted ranks are 0..nacc-1
            const int at = sBase + rk;
            ws.entry[at] = make_int2((int)q, __float_as_int(ws.row_max[q]));
            ws.key[at] = 0ull;
            ws.done[at] = 0;
        }
        accept_mask[q] = acc ? 1 : 0;
        if (!read_only) {
            if (!acc)
                canvas[q] = (int32_t)dg::random_token(seed, p.request_id, (uint32_t)p.step, (uint32_t)i,
                                                      dg::kStreamRenoise, (uint32_t)V);
            else if (!deferred)
                canvas[q] = sample[q];
        }
        prev_argmax[q] = am;
    }
    if (i == 0) {
        const int32_t st = same ? st0 + 1 : 0;
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
// LM head: each row's statistics from the softmax states the GEMM epilogue recorded per
// 256-column tile (same quantities as RowState, records [tile][5][R]).  One CTA per 32
// consecutive rows (lane = row, so every load is 128 contiguous bytes); its 32 warps take the
// tiles in 32 contiguous ranges and are merged in warp order, so the result does not depend
// on timing.  Writes what k1_row_stats writes for a canvas without DG_SAMPLE_ALL (sample -1,
// the row's maximum for the deferred sampler) and clears the list of accepted rows.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) k_lm_stats_merge(
    const float* __restrict__ rec, int64_t R, int32_t n_tiles, int32_t L, const dg_canvas_params* __restrict__ params,
    int32_t* __restrict__ argmax_out, int32_t* __restrict__ sample_out, float* __restrict__ entropy_out,
    float* __restrict__ lse_out, DeferredWs ws, unsigned* status) {
    __shared__ RowState part[32][33];
    __shared__ int part_bad[32][33];
    dg::pdl_wait();
    dg::pdl_release();
    if (ws.count && blockIdx.x == 0 && threadIdx.x == 0) *ws.count = 0;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t row = (int64_t)blockIdx.x * 32 + lane;
    const int64_t canvas = row < R ? row / L : 0;
    const dg_canvas_params p = params[canvas];
    const bool t_ok = p.temperature > 0.f && isfinite(p.temperature);
    const bool use = row < R && (p.flags & DG_ACTIVE) && t_ok;
    const float invT = use ? 1.0f / p.temperature : 1.f;
    const float k2 = kLog2e * invT;
    RowState st{-INFINITY, 0.f, 0.f, 0.f, 0x7fffffff};
    bool bad = false;
    if (use) {
        const int t0 = (int)((int64_t)warp * n_tiles / 32), t1 = (int)((int64_t)(warp + 1) * n_tiles / 32);
        constexpr int kB = 4;  // records in flight per thread
        for (int t = t0; t < t1; t += kB) {
            float f[kB][5];
#pragma unroll
            for (int b = 0; b < kB; ++b) {
                if (t + b < t1) {
                    const float* q = rec + (int64_t)(t + b) * 5 * R + row;
#pragma unroll
                    for (int k = 0; k < 5; ++k) f[b][k] = __ldcs(q + k * R);
                }
            }
#pragma unroll
            for (int b = 0; b < kB; ++b) {
                if (t + b < t1) {
                    if (f[b][1] != f[b][1]) {
                        bad = true;
                    } else {
                        st = merge(st, RowState{f[b][0], f[b][1], f[b][2], f[b][3], __float_as_int(f[b][4])}, k2);
                    }
                }
            }
        }
    }
    part[warp][lane] = st;
    part_bad[warp][lane] = bad ? 1 : 0;
    __syncthreads();
    if (warp != 0) return;
    if (row < R && (p.flags & DG_ACTIVE) && !t_ok) {
        if (row % L == 0) dg::raise_status(status, DG_DEV_BAD_PARAM);
        return;
    }
    if (!use) return;
    RowState rs = part[0][lane];
    for (int w = 1; w < 32; ++w) {
        rs = merge(rs, part[w][lane], k2);
        bad |= part_bad[w][lane] != 0;
    }
    const bool empty = rs.m == -INFINITY;
    const bool row_bad = bad || rs.m == INFINITY || !isfinite(rs.r) || !isfinite(rs.t);
    const float sum = rs.c + rs.r;
    const float lns = (rs.c == 1.f) ? log1pf(rs.r) : logf(rs.c) + log1pf(rs.r / rs.c);
    entropy_out[row] = lns - rs.t * kLn2 / sum;
    lse_out[row] = rs.m * invT + lns;
    argmax_out[row] = empty ? 0 : rs.idx;
    sample_out[row] = -1;
    ws.row_max[row] = (empty || row_bad) ? __int_as_float(0x7fc00000) : rs.m;
    if (row_bad) dg::raise_status(status, DG_DEV_NAN_INF_ROW);
    if (empty) dg::raise_status(status, DG_DEV_EMPTY_ROW);
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

// Statistics of every active row (+ samples of DG_SAMPLE_ALL canvases); clears the list.
template <int DT>
dg_status launch_k1(const void* logits, int64_t ld, int64_t n, int32_t L, int64_t V,
                    const dg_canvas_params* params, uint64_t seed, int32_t* argmax, int32_t* sample, float* entropy,
                    float* lse, const DeferredWs& ws, const ChoiceOut& co, cudaStream_t stream) {
    auto kern = k1_row_stats<DT>;
    const size_t smem = k1_smem_bytes<DT>();
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return DG_ERR_CUDA;
    const int64_t ld_bytes = ld * (DT == 0 ? 2 : 4);
    const cudaError_t e = dghost::launch_pdl(kern, dim3((unsigned)L, (unsigned)n, 1), dim3(kK1Threads), smem, stream,
                                             static_cast<const unsigned char*>(logits), ld_bytes, V, L, params, seed,
                                             argmax, sample, entropy, lse, ws, co, dghost::status_word());
    dghost::count_launch();
    return dghost::cuda_status(e);
}

// Samples and tokens of the listed accepted rows (the list length is only known on the
// device): in line, 3 CTAs of kDWarps warps per SM; beside (for another stream), one CTA of
// kSideWarps warps per SM, small enough to share an SM with a GEMM CTA.
template <int DT>
dg_status launch_kd(const void* logits, int64_t ld, int64_t n, int32_t L, int64_t V,
                    const dg_canvas_params* params, uint64_t seed, const DeferredWs& ws, int32_t* sample,
                    int32_t* canvas, bool beside, cudaStream_t stream) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return DG_ERR_CUDA;
    const int64_t cpr = (V * (DT == 0 ? 2 : 4) + kChunkBytes - 1) / kChunkBytes;
    const int64_t max_items = n * (int64_t)L * cpr;
    const int warps = beside ? kSideWarps : kDWarps;
    const unsigned grid = (unsigned)std::max<int64_t>(
        1, std::min<int64_t>((int64_t)(beside ? 1 : 3) * sms, (max_items + warps - 1) / warps));
    const int64_t ld_bytes = ld * (DT == 0 ? 2 : 4);
    // few rows (a single request): contiguous runs per warp; else single chunks
    const bool runs = n * (int64_t)L <= kRunsMaxRows;
    auto kern = beside ? (runs ? k1_sample_listed<DT, true, kSideWarps> : k1_sample_listed<DT, false, kSideWarps>)
                       : (runs ? k1_sample_listed<DT, true, kDWarps> : k1_sample_listed<DT, false, kDWarps>);
    const cudaError_t e = dghost::launch_pdl(kern, dim3(grid), dim3(warps * 32), 0, stream,
                                             static_cast<const unsigned char*>(logits), ld_bytes, V, L, params, seed,
                                             ws, sample, canvas, n * (int64_t)L);
    dghost::count_launch();
    return dghost::cuda_status(e);
}

dg_status launch_k2(const float* entropy, const int32_t* sample, const int32_t* argmax, int64_t n, int32_t L,
                    int64_t V, const dg_canvas_params* params, uint64_t seed, int32_t* canvas, int32_t* prev_argmax,
                    int32_t* stable_count, uint8_t* accept_mask, uint8_t* converged, float* mean_entropy,
                    int32_t* n_accept, const DeferredWs& ws, cudaStream_t stream, bool late_release = false) {
    const unsigned threads = (unsigned)((L + 31) / 32 * 32);
    auto kern = threads <= 256 ? k2_accept<256> : k2_accept<1024>;
    const cudaError_t e = dghost::launch_pdl(kern, dim3((unsigned)n), dim3(threads), 0, stream, entropy, sample,
                                             argmax, L, V, params, seed, canvas, prev_argmax, stable_count,
                                             accept_mask, converged, mean_entropy, n_accept, ws,
                                             late_release ? 1 : 0, dghost::status_word());
    dghost::count_launch();
    return dghost::cuda_status(e);
}

// The deferred-sampling workspace: a count (padded to 256 bytes), then per listed row an
// entry (8 bytes), a key (8) and a chunk counter (4), and per row its maximum (4).
size_t denoise_ws_bytes(int64_t rows) { return (size_t)256 + (size_t)rows * 24; }

DeferredWs carve_ws(void* workspace, int64_t rows) {
    unsigned char* b = static_cast<unsigned char*>(workspace);
    DeferredWs ws;
    ws.count = reinterpret_cast<int32_t*>(b);
    ws.entry = reinterpret_cast<int2*>(b + 256);
    ws.key = reinterpret_cast<unsigned long long*>(b + 256 + 8 * rows);
    ws.done = reinterpret_cast<int32_t*>(b + 256 + 16 * rows);
    ws.row_max = reinterpret_cast<float*>(b + 256 + 20 * rows);
    ws.all_deferred = 0;
    return ws;
}

// LM-head workspace: the deferred-sampling workspace, the list of active canvases, then the
// per-tile softmax states (5 floats per row and 256-column tile).
struct LmLayout {
    size_t plan, rec, total;
    int32_t n_tiles;
};

LmLayout lm_layout(int64_t n, int32_t L, int64_t V) {
    const int64_t rows = n * (int64_t)L;
    LmLayout l;
    l.n_tiles = (int32_t)((V + dghost::kLmTileCols - 1) / dghost::kLmTileCols);
    l.plan = (denoise_ws_bytes(rows) + 255) / 256 * 256;
    l.rec = l.plan + ((size_t)(n + 1) * 4 + 255) / 256 * 256;
    l.total = l.rec + ((size_t)rows * l.n_tiles * 5 * 4 + 255) / 256 * 256;
    return l;
}

// Shapes, strides and alignment shared by the LM-head entry points.
dg_status lm_head_check(const void* hidden, int64_t ldh, const void* W, int64_t ldw, int64_t n, int32_t L, int64_t V,
                        int32_t d, const void* params, const void* logits, int64_t ld, const void* workspace,
                        size_t workspace_bytes) {
    dg_status s = check_canvas_dims(n, L, V);
    if (s != DG_OK) return s;
    if (d < 8 || d > 65536 || (d % 8) || ldh < d || ldw < d || ld < V || V >= (1LL << 30)) return DG_ERR_INVALID_ARG;
    if (n == 0) return DG_OK;
    if (!hidden || !W || !params || !logits) return DG_ERR_INVALID_ARG;
    if (!aligned16(hidden) || !aligned16(W) || !aligned16(logits) || (ldh % 8) || (ldw % 8) || (ld % 8))
        return DG_ERR_ALIGNMENT;
    if (!workspace || workspace_bytes < lm_layout(n, L, V).total) return DG_ERR_WORKSPACE;
    if (!aligned16(workspace)) return DG_ERR_ALIGNMENT;
    return DG_OK;
}

}  // namespace

extern "C" {

size_t dg_denoise_workspace_bytes(int64_t n_canvas, int32_t L, int64_t, dg_dtype) {
    if (n_canvas < 0 || L < 0) return 0;
    return (denoise_ws_bytes(n_canvas * (int64_t)L) + 255) / 256 * 256;
}

static dg_status denoise_stats(const void* logits, dg_dtype dtype, int64_t ld, int64_t n_canvas, int32_t L,
                               int64_t V, const dg_canvas_params* params, uint64_t seed, int32_t* canvas,
                               int32_t* prev_argmax, int32_t* stable_count, uint8_t* accept_mask, int32_t* argmax,
                               int32_t* sample, float* entropy, float* lse, uint8_t* converged, float* mean_entropy,
                               int32_t* n_accept, const ChoiceOut& co, void* workspace, size_t workspace_bytes,
                               dg_stream_t stream) {
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
    if (!workspace || workspace_bytes < dg_denoise_workspace_bytes(n_canvas, L, V, dtype)) return DG_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 7u) != 0) return DG_ERR_ALIGNMENT;
    const DeferredWs ws = carve_ws(workspace, n_canvas * (int64_t)L);
    cudaStream_t st = (cudaStream_t)stream;
    s = dtype == DG_BF16
            ? launch_k1<0>(logits, ld, n_canvas, L, V, params, seed, argmax, sample, entropy, lse, ws, co, st)
            : launch_k1<1>(logits, ld, n_canvas, L, V, params, seed, argmax, sample, entropy, lse, ws, co, st);
    if (s != DG_OK) return s;
    return launch_k2(entropy, sample, argmax, n_canvas, L, V, params, seed, canvas, prev_argmax, stable_count,
                     accept_mask, converged, mean_entropy, n_accept, ws, st);
}

dg_status dg_denoise_stats(const void* logits, dg_dtype dtype, int64_t ld, int64_t n_canvas, int32_t L, int64_t V,
                           const dg_canvas_params* params, uint64_t seed, int32_t* canvas, int32_t* prev_argmax,
                           int32_t* stable_count, uint8_t* accept_mask, int32_t* argmax, int32_t* sample,
                           float* entropy, float* lse, uint8_t* converged, float* mean_entropy, int32_t* n_accept,
                           void* workspace, size_t workspace_bytes, dg_stream_t stream) {
    return denoise_stats(logits, dtype, ld, n_canvas, L, V, params, seed, canvas, prev_argmax, stable_count,
                         accept_mask, argmax, sample, entropy, lse, converged, mean_entropy, n_accept, ChoiceOut{},
                         workspace, workspace_bytes, stream);
}

dg_status dg_denoise_row_stats(const void* logits, dg_dtype dtype, int64_t ld, int64_t n_canvas, int32_t L, int64_t V,
                               const dg_canvas_params* params, uint64_t seed, int32_t* argmax, int32_t* sample,
                               float* entropy, float* lse, void* workspace, size_t workspace_bytes,
                               dg_stream_t stream) {
    if (dtype != DG_BF16 && dtype != DG_FP32) return DG_ERR_INVALID_ARG;
    dg_status s = check_canvas_dims(n_canvas, L, V);
    if (s != DG_OK) return s;
    if (ld < V) return DG_ERR_INVALID_ARG;
    if (n_canvas == 0) return DG_OK;
    if (!logits || !params || !argmax || !sample || !entropy || !lse) return DG_ERR_INVALID_ARG;
    const int64_t es = dtype == DG_BF16 ? 2 : 4;
    if (!aligned16(logits) || (ld * es) % 16 != 0) return DG_ERR_ALIGNMENT;
    if (!k1_supported(dtype, V)) return DG_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < dg_denoise_workspace_bytes(n_canvas, L, V, dtype)) return DG_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 7u) != 0) return DG_ERR_ALIGNMENT;
    const DeferredWs ws = carve_ws(workspace, n_canvas * (int64_t)L);
    cudaStream_t st = (cudaStream_t)stream;
    return dtype == DG_BF16
               ? launch_k1<0>(logits, ld, n_canvas, L, V, params, seed, argmax, sample, entropy, lse, ws, ChoiceOut{}, st)
               : launch_k1<1>(logits, ld, n_canvas, L, V, params, seed, argmax, sample, entropy, lse, ws, ChoiceOut{}, st);
}

dg_status dg_denoise_accept(const float* entropy, const int32_t* sample, const int32_t* argmax, int64_t n_canvas,
                            int32_t L, int64_t V, const dg_canvas_params* params, uint64_t seed, int32_t* canvas,
                            int32_t* prev_argmax, int32_t* stable_count, uint8_t* accept_mask, uint8_t* converged,
                            float* mean_entropy, int32_t* n_accept, void* workspace, size_t workspace_bytes,
                            dg_stream_t stream) {
    dg_status s = check_canvas_dims(n_canvas, L, V);
    if (s != DG_OK) return s;
    if (n_canvas == 0) return DG_OK;
    if (!entropy || !sample || !argmax || !params || !canvas || !prev_argmax || !stable_count || !accept_mask ||
        !converged)
        return DG_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < dg_denoise_workspace_bytes(n_canvas, L, V, DG_BF16)) return DG_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 7u) != 0) return DG_ERR_ALIGNMENT;
    const DeferredWs ws = carve_ws(workspace, n_canvas * (int64_t)L);
    return launch_k2(entropy, sample, argmax, n_canvas, L, V, params, seed, canvas, prev_argmax, stable_count,
                     accept_mask, converged, mean_entropy, n_accept, ws, (cudaStream_t)stream, true);
}

static dg_status denoise_samples(const void* logits, dg_dtype dtype, int64_t ld, int64_t n_canvas, int32_t L,
                                 int64_t V, const dg_canvas_params* params, uint64_t seed, int32_t* canvas,
                                 int32_t* sample, void* workspace, size_t workspace_bytes, bool beside,
                                 cudaStream_t st) {
    if (dtype != DG_BF16 && dtype != DG_FP32) return DG_ERR_INVALID_ARG;
    dg_status s = check_canvas_dims(n_canvas, L, V);
    if (s != DG_OK) return s;
    if (ld < V) return DG_ERR_INVALID_ARG;
    if (n_canvas == 0) return DG_OK;
    if (!logits || !params || !canvas || !sample) return DG_ERR_INVALID_ARG;
    const int64_t es = dtype == DG_BF16 ? 2 : 4;
    if (!aligned16(logits) || (ld * es) % 16 != 0) return DG_ERR_ALIGNMENT;
    if (!k1_supported(dtype, V)) return DG_ERR_UNSUPPORTED;
    if (!workspace || workspace_bytes < dg_denoise_workspace_bytes(n_canvas, L, V, dtype)) return DG_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 7u) != 0) return DG_ERR_ALIGNMENT;
    const DeferredWs ws = carve_ws(workspace, n_canvas * (int64_t)L);
    return dtype == DG_BF16
               ? launch_kd<0>(logits, ld, n_canvas, L, V, params, seed, ws, sample, canvas, beside, st)
               : launch_kd<1>(logits, ld, n_canvas, L, V, params, seed, ws, sample, canvas, beside, st);
}

dg_status dg_denoise_samples(const void* logits, dg_dtype dtype, int64_t ld, int64_t n_canvas, int32_t L, int64_t V,
                             const dg_canvas_params* params, uint64_t seed, int32_t* canvas, int32_t* sample,
                             void* workspace, size_t workspace_bytes, dg_stream_t stream) {
    return denoise_samples(logits, dtype, ld, n_canvas, L, V, params, seed, canvas, sample, workspace,
                           workspace_bytes, true, (cudaStream_t)stream);
}

dg_status dg_denoise_step(const void* logits, dg_dtype dtype, int64_t ld, int64_t n_canvas, int32_t L, int64_t V,
                          const dg_canvas_params* params, uint64_t seed, int32_t* canvas, int32_t* prev_argmax,
                          int32_t* stable_count, uint8_t* accept_mask, int32_t* argmax, int32_t* sample,
                          float* entropy, float* lse, uint8_t* converged, float* mean_entropy, int32_t* n_accept,
                          void* workspace, size_t workspace_bytes, dg_stream_t stream) {
    dg_status s = denoise_stats(logits, dtype, ld, n_canvas, L, V, params, seed, canvas, prev_argmax, stable_count,
                                accept_mask, argmax, sample, entropy, lse, converged, mean_entropy, n_accept,
                                ChoiceOut{}, workspace, workspace_bytes, stream);
    if (s != DG_OK || n_canvas == 0) return s;
    // alone on its stream: three CTAs of 8 warps per SM hide more of the load latency
    return denoise_samples(logits, dtype, ld, n_canvas, L, V, params, seed, canvas, sample, workspace,
                           workspace_bytes, false, (cudaStream_t)stream);
}

dg_status dg_denoise_step_choices(const void* logits, dg_dtype dtype, int64_t ld, int64_t n_canvas, int32_t L,
                                  int64_t V, const dg_canvas_params* params, uint64_t seed, int32_t* canvas,
                                  int32_t* prev_argmax, int32_t* stable_count, uint8_t* accept_mask, int32_t* argmax,
                                  int32_t* sample, float* entropy, float* lse, uint8_t* converged,
                                  float* mean_entropy, int32_t* n_accept, const int32_t* choices, int32_t C,
                                  float* probs, void* workspace, size_t workspace_bytes, dg_stream_t stream) {
    if (C < 1 || C > 1024) return DG_ERR_INVALID_ARG;
    if (n_canvas > 0 && (!choices || !probs)) return DG_ERR_INVALID_ARG;
    dg_status s = denoise_stats(logits, dtype, ld, n_canvas, L, V, params, seed, canvas, prev_argmax, stable_count,
                                accept_mask, argmax, sample, entropy, lse, converged, mean_entropy, n_accept,
                                ChoiceOut{choices, probs, C}, workspace, workspace_bytes, stream);
    if (s != DG_OK || n_canvas == 0) return s;
    return denoise_samples(logits, dtype, ld, n_canvas, L, V, params, seed, canvas, sample, workspace,
                           workspace_bytes, false, (cudaStream_t)stream);
}

size_t dg_lm_head_workspace_bytes(int64_t n_canvas, int32_t L, int64_t V) {
    if (n_canvas < 0 || L < 0 || V < 0) return 0;
    return lm_layout(n_canvas, L, V).total;
}

dg_status dg_lm_head_logits(const uint16_t* hidden, int64_t ldh, const uint16_t* W_lm, int64_t ldw, int64_t n_canvas,
                            int32_t L, int64_t V, int32_t d, const dg_canvas_params* params, uint16_t* logits,
                            int64_t ld, void* workspace, size_t workspace_bytes, dg_stream_t stream) {
    const dg_status s = lm_head_check(hidden, ldh, W_lm, ldw, n_canvas, L, V, d, params, logits, ld, workspace,
                                      workspace_bytes);
    if (s != DG_OK || n_canvas == 0) return s;
    const LmLayout lay = lm_layout(n_canvas, L, V);
    unsigned char* b = static_cast<unsigned char*>(workspace);
    return dghost::lm_head_gemm(hidden, ldh, W_lm, ldw, n_canvas, L, V, d, params, logits, ld,
                                reinterpret_cast<int32_t*>(b + lay.plan), nullptr, (cudaStream_t)stream);
}

dg_status dg_lm_head_denoise_step(const uint16_t* hidden, int64_t ldh, const uint16_t* W_lm, int64_t ldw,
                                  int64_t n_canvas, int32_t L, int64_t V, int32_t d, const dg_canvas_params* params,
                                  uint64_t seed, uint16_t* logits, int64_t ld, int32_t* canvas, int32_t* prev_argmax,
                                  int32_t* stable_count, uint8_t* accept_mask, int32_t* argmax, int32_t* sample,
                                  float* entropy, float* lse, uint8_t* converged, float* mean_entropy,
                                  int32_t* n_accept, void* workspace, size_t workspace_bytes, dg_stream_t stream) {
    dg_status s = lm_head_check(hidden, ldh, W_lm, ldw, n_canvas, L, V, d, params, logits, ld, workspace,
                                workspace_bytes);
    if (s != DG_OK || n_canvas == 0) return s;
    if (!canvas || !prev_argmax || !stable_count || !accept_mask || !argmax || !sample || !entropy || !lse ||
        !converged)
        return DG_ERR_INVALID_ARG;
    const LmLayout lay = lm_layout(n_canvas, L, V);
    unsigned char* b = static_cast<unsigned char*>(workspace);
    const int64_t R = n_canvas * (int64_t)L;
    float* rec = reinterpret_cast<float*>(b + lay.rec);
    cudaStream_t st = (cudaStream_t)stream;
    s = dghost::lm_head_gemm(hidden, ldh, W_lm, ldw, n_canvas, L, V, d, params, logits, ld,
                             reinterpret_cast<int32_t*>(b + lay.plan), rec, st);
    if (s != DG_OK) return s;
    DeferredWs ws = carve_ws(workspace, R);
    ws.all_deferred = 1;
    const cudaError_t e = dghost::launch_pdl(k_lm_stats_merge, dim3((unsigned)((R + 31) / 32)), dim3(1024), 0, st, rec,
                                             R, lay.n_tiles, L, params, argmax, sample, entropy, lse, ws,
                                             dghost::status_word());
    dghost::count_launch();
    if (e != cudaSuccess) return DG_ERR_CUDA;
    s = launch_k2(entropy, sample, argmax, n_canvas, L, V, params, seed, canvas, prev_argmax, stable_count,
                  accept_mask, converged, mean_entropy, n_accept, ws, st);
    if (s != DG_OK) return s;
    return launch_kd<0>(logits, ld, n_canvas, L, V, params, seed, ws, sample, canvas, false, st);
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
                     accept_mask, converged, mean_entropy, n_accept, DeferredWs{}, (cudaStream_t)stream);
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
