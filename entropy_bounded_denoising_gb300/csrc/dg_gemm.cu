// dg_gemm.cu -- tensor-core GEMM engine (tcgen05 + TMEM + TMA, sm_103a) and the
// self-conditioning feedback built on it.
//
// Method (DiffusionGemma vLLM page, "DiffusionGemma: vLLM이 네이티브로 지원하는 최초의 디퓨전
// 언어 모델(dLLM)", section "자기 조건화" (self-conditioning), and the state paragraph of
// "DiffusionGemmaModelState와 DiffusionSampler"): the step's softmax P becomes the
// probability-weighted mean of the token embeddings, pe = P . E, which a small gated MLP
// turns into the feedback added to the next pass's canvas embeddings; the feedback is zero
// for the encoder prefill and commit passes.  The MLP form (no bias, GELU-tanh gate) is a
// reading; the pages only say "small gated MLP".
//
// Engine (one CTA per SM, persistent, warp-specialised):
//   warp 0      TMA producer: A and B tiles into a ring of shared-memory stages;
//   warp 1      tcgen05.mma issuer (one elected thread) and TMEM owner;
//   warps 2..5  epilogue: TMEM -> registers -> global (tcgen05.ld), one TMEM lane quarter each;
//   warps 6..13 (softmax A only) transform: the logits tile landed by TMA is turned in place
//               into P = exp2(x * log2e / T - lse * log2e) in bf16, so P never leaves the SM;
//               two groups of four warps take the stages in turn.
// Work items are (k-slice, n-tile, m-tile) with the m-tile fastest; item w runs on CTA
// w mod P in round w / P.  All CTAs of a round therefore stream the same k-range, and the
// B tile (embedding rows) and A tile (logit rows) they share are read from HBM once and
// served from L2 to the others.  With more than one k-slice the fp32 partial tiles go to a
// workspace slot per item and a fix-up kernel adds them in slice order (deterministic).
#include <cuda.h>
#include <cuda_runtime.h>

#include <math.h>

#include <algorithm>
#include <mutex>

#include <cooperative_groups.h>

#include "dg_common.cuh"

namespace cg = cooperative_groups;

namespace {

constexpr int BM = 128;
constexpr float kLog2e = 1.4426950408889634f;

// A_TMA_CANVAS: plain bf16 A rows per canvas ([n][L][ld], 3D map), as the LM head reads the
// hidden states of the listed canvases
enum AMode { A_TMA = 0, A_SOFTMAX_BF16 = 1, A_SOFTMAX_FP32 = 2, A_TMA_CANVAS = 3 };
enum BMode { B_KMAJOR = 0, B_MNMAJOR = 1, B_KMAJOR_GATEUP = 2 };
enum Epi { EPI_F32 = 0, EPI_BF16 = 1, EPI_GELU_GATEUP = 2, EPI_SCATTER_BF16 = 3, EPI_LOGIT_STATS = 4 };

constexpr int kSplitTab = 256;

struct GemmArgs {
    int32_t m_tiles;        // m-tiles when plan == nullptr; upper bound otherwise
    const int32_t* plan;    // plan[0] = active canvases, plan[1..] = their ids (or nullptr)
    int32_t tpc;            // m-tiles per canvas
    int32_t n_tiles;
    int32_t k_blocks;
    int32_t splits;         // k-slices
    int64_t K;              // true K extent (tail masking of the softmax operand)
    int32_t L;              // rows per canvas
    const float* lse;       // [n_canvas][L]
    const dg_canvas_params* params;
    int32_t epi;
    void* out;
    int64_t ldo;            // output row stride in elements
    int32_t n_valid;        // valid output columns
    int32_t m_valid;        // valid output rows (plain GEMMs)
    float* partial;         // [items][BM * BN] when splits > 1
    unsigned* status;
    // dyn_splits = 1: the k-slices are chosen on the device from the active m-tiles (the host
    // only knows an upper bound when a plan lists the rows), the same way in the GEMM and its
    // fix-up, from these values of the host's plan
    int32_t dyn_splits;
    int32_t cm_plan;        // CTAs per cluster
    int32_t clusters;       // concurrent clusters
    int32_t min_slice;      // k-blocks
    int64_t max_slots;      // partial tiles the workspace holds
    int32_t split_below;    // split only below this round efficiency (percent)
    // P.E: a counter of work items whose loads the CTAs' producers have issued (zeroed by
    // the plan launch), used to keep the clusters' items in step (see pace_wait); null: none
    unsigned* pace;
    // the same rule tabulated by the host for plans listing j <= kSplitTab canvases
    // (split_tab[j]); larger plans evaluate it on the device
    uint8_t split_tab[260];
    // EPI_LOGIT_STATS: per (tile column block, row) softmax states, [n_tiles][5][stats_rows]
    float* stats;
    int64_t stats_rows;
};

// k-slices: the fewest that keep the rounds at least 95 % full, with slices of at least
// `min_slice` k-blocks so that the partial tiles stay cheap next to the MMA work.  Round
// efficiencies items / (rounds * P) are compared as exact fractions (integer arithmetic:
// host and device agree, and GB300's slow FP64 stays out of every CTA's prologue).
__host__ __device__ inline int choose_splits(int64_t T, int k_blocks, int P, int min_slice) {
    int best = 1;
    int64_t best_num = 0, best_den = 1;
    for (int s = 1; s <= 32; ++s) {
        if (s > 1 && k_blocks / s < min_slice) break;
        const int64_t items = T * s;  // < 2^31 for every supported shape: 32-bit division
        const int64_t den = (int64_t)(((uint32_t)items + (uint32_t)P - 1u) / (uint32_t)P) * P;
        if (items * best_den > best_num * den) {
            best_num = items;
            best_den = den;
            best = s;
        }
        if (items * 100 >= den * 95) break;
    }
    return best;
}

// The k-slices for `mt` m-tiles (`per_split` work groups per slice): per the plan's rule
// (round efficiency below split_below percent, within max_slots partial tiles).
__host__ __device__ inline int plan_splits(int64_t per_split, int64_t mt, int n_tiles, int k_blocks, int clusters,
                                           int min_slice, int64_t max_slots, int split_below) {
    if (per_split <= 0 || clusters <= 0) return 1;
    const int64_t den1 = (int64_t)(((uint32_t)per_split + (uint32_t)clusters - 1u) / (uint32_t)clusters) * clusters;
    int splits = per_split * 100 < (int64_t)split_below * den1
                     ? choose_splits(per_split, k_blocks, clusters, min_slice < 1 ? 1 : min_slice)
                     : 1;
    while (splits > 1 && mt * n_tiles * splits > max_slots) --splits;
    return splits;
}

// PAIR_: the CTA pair of a 2-CTA cluster computes one 256-row tile with cta_group::2 MMAs;
// each CTA then holds half of every 256-column B slab (for the gate/up tile: the first CTA
// the gate rows, the second the up rows).
template <int AM, int BMD, int BN_, int BK_, int STAGES_, bool PAIR_ = false>
struct Cfg {
    static constexpr bool kPair = PAIR_;
    static constexpr int kAMode = AM;
    static constexpr int kBMode = BMD;
    static constexpr int BN = BN_;
    static constexpr int BK = BK_;
    static constexpr int STAGES = STAGES_;
    static constexpr bool kXform = AM == A_SOFTMAX_BF16 || AM == A_SOFTMAX_FP32;
    static constexpr int kAccCols = BN;                      // fp32 accumulator columns
    static constexpr int kNAcc = (BN <= 256) ? 2 : 1;        // double-buffered when it fits
    static constexpr int kTmemCols = kAccCols * kNAcc;       // 256 or 512
    static constexpr int kXformThreads = 256;                // DG_XFORM_GROUPS groups taking stages in turn
    static constexpr int kXformWarps = kXformThreads / 32;
    static constexpr int kThreads = kXform ? 192 + kXformThreads : 192;
    static constexpr int kATileBytes = BM * BK * 2;
    static constexpr int kStageBytesFp32 = (AM == A_SOFTMAX_FP32) ? BM * BK * 4 : 0;
    static constexpr int kBTileBytes = BK * BN * 2 / (PAIR_ ? 2 : 1);  // this CTA's part of the B tile
    static constexpr int kStageBytes = kATileBytes + kBTileBytes + kStageBytesFp32;
    static constexpr int kASwizzle = BK * 2;                 // 64 or 128 bytes: one swizzle row per tile row
    static constexpr uint32_t kTxBytes = (uint32_t)(kBTileBytes + (AM == A_SOFTMAX_FP32 ? kStageBytesFp32 : kATileBytes));
    static constexpr size_t kSmem = 1024 + (size_t)STAGES * kStageBytes + 1024;
    static_assert(!PAIR_ || (BMD == B_MNMAJOR ? BN_ == 512 : BN_ == 256), "pair mode: BN 512 (N-major B) or 256");
    static_assert(STAGES_ <= 12, "stage barriers");
    static_assert(kSmem <= 232448, "fits the opt-in shared memory of an SM");
};

// ------------------------------------------------------------------ descriptors
using dg::instr_desc;
using dg::smem_desc;

// ------------------------------------------------------------------ scheduling
struct Item {
    int m, n, kb_lo, kb_hi;
    int m_load;   // m-tile whose rows are loaded (a real tile even for padding members)
    bool valid;   // false for the padding members of the last group of m-tiles
    int64_t w;    // partial-tile slot: k-slice * T + n * mt + m
};

DG_DEVINL int active_m_tiles(const GemmArgs& a) {
    if (!a.plan) return a.m_tiles;
    return min(a.m_tiles, a.plan[0] * a.tpc);
}

// Work is cut into groups of `cm` consecutive m-tiles sharing one (k-slice, n-tile); the cm
// CTAs of a cluster run a group together (rank r takes m-tile mg * cm + r) so that they can
// share the B tile.  Groups are ordered (k-slice, n-tile, m-group), m fastest.
DG_DEVINL int64_t group_count(const GemmArgs& a, int mt, int cm, int splits) {
    return (int64_t)splits * a.n_tiles * ((mt + cm - 1) / cm);
}

// The launch's k-slices for `mt` active m-tiles.  The rule's loop of integer divisions takes
// microseconds on one thread, so plans of up to kSplitTab canvases read the host's table.
DG_DEVINL int active_splits(const GemmArgs& a, int mt) {
    if (!a.dyn_splits) return a.splits;
    if (a.plan && mt % a.tpc == 0 && mt / a.tpc <= kSplitTab) return a.split_tab[mt / a.tpc];
    const int64_t per_split = (int64_t)a.n_tiles * ((mt + a.cm_plan - 1) / a.cm_plan);
    return plan_splits(per_split, mt, a.n_tiles, a.k_blocks, a.clusters, a.min_slice, a.max_slots, a.split_below);
}

// Group counts stay far below 2^32 (k-slices x n-tiles x m-groups), so the indices are split
// in 32-bit arithmetic: a 64-bit division is a long emulated sequence, paid by every warp role
// before its first item.
DG_DEVINL Item decode(const GemmArgs& a, int mt, int cm, int rank, int64_t G, int splits) {
    const uint32_t mgc = (uint32_t)((mt + cm - 1) / cm);
    const uint32_t per_s = (uint32_t)a.n_tiles * mgc;
    const uint32_t g = (uint32_t)G;
    const int s = (int)(g / per_s);
    const uint32_t rem = g - (uint32_t)s * per_s;
    Item it;
    it.n = (int)(rem / mgc);
    it.m = (int)(rem - (uint32_t)it.n * mgc) * cm + rank;
    it.valid = it.m < mt;
    it.m_load = it.valid ? it.m : mt - 1;
    // (s + 1) * k_blocks <= 33 * 2^26 < 2^32: unsigned 32-bit
    it.kb_lo = (int)((uint32_t)s * (uint32_t)a.k_blocks / (uint32_t)splits);
    it.kb_hi = (int)((uint32_t)(s + 1) * (uint32_t)a.k_blocks / (uint32_t)splits);
    it.w = (int64_t)s * mt * a.n_tiles + (int64_t)it.n * mt + it.m;
    return it;
}

// Keeps the clusters of a persistent P.E launch in step: before loading its item j, a CTA's
// producer waits until every CTA has issued the loads of its item j - 1 (items go round-robin,
// so if any cluster has an item j every cluster had items 0 .. j - 1).  Items of one round
// share their logits and embedding k-blocks through L2 only while the clusters stream them at
// about the same time; left alone, they drift apart over a launch and most re-reads miss.
// Only the timing depends on it: an expired wait raises DG_DEV_TIMEOUT and goes on.
#ifndef DG_PE_PACE
#define DG_PE_PACE 1
#endif
DG_DEVINL void pace_wait(const unsigned* ctr, unsigned target, unsigned* status) {
    for (uint32_t i = 0; i < (1u << 20); ++i) {
        if (*(volatile const unsigned*)ctr >= target) return;
        __nanosleep(128);
    }
    dg::raise_status(status, DG_DEV_TIMEOUT);
}

DG_DEVINL int canvas_of(const GemmArgs& a, int m) {
    const int j = m / a.tpc;
    return a.plan ? a.plan[1 + j] : j;
}

DG_DEVINL uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

DG_DEVINL float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// GELU, tanh form: 0.5 z (1 + tanh y), y = sqrt(2 / pi) (z + 0.044715 z^3), evaluated as
// z * sigmoid(2 y) = z / (1 + 2^(-2 y log2 e)) (the same function, since 1 + tanh y =
// 2 / (1 + e^(-2 y))): one exponential and one reciprocal, about 1e-6 relative, far inside the
// bf16 rounding of the hidden layer.  Large |z|: the exponential saturates to 0 or inf and the
// result to z or -0.
DG_DEVINL float gelu_tanh(float z) {
    const float k2 = -2.f * 0.7978845608028654f * 1.4426950408889634f;  // -2 sqrt(2 / pi) log2 e
    float e, r;
    const float t = k2 * (z + 0.044715f * z * z * z);
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(t));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + e));
    return z * r;
}

// Groups of softmax-transform threads that take the P.E stages in turn (2: measured fastest
// against 1, 4 and 8 on the batched workload; see the transform loop).
#ifndef DG_XFORM_GROUPS
#define DG_XFORM_GROUPS 2
#endif

constexpr int kMaxStages = 12;

struct __align__(8) GemmShared {
    uint64_t full[kMaxStages];
    uint64_t xform[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t accf[2];
    uint64_t acce[2];
    uint32_t tmem_base;
    int abort_flag;
    int splits;  // k-slices of this launch
};

DG_DEVINL bool aborted(const GemmShared& sh) { return *(volatile const int*)&sh.abort_flag != 0; }

// Warp-uniform form for loops whose body holds whole-warp operations.
DG_DEVINL bool aborted_warp(const GemmShared& sh) { return __shfl_sync(0xffffffffu, (int)aborted(sh), 0) != 0; }

DG_DEVINL void do_abort(GemmShared& sh, unsigned* status) {
    *(volatile int*)&sh.abort_flag = 1;
    dg::raise_status(status, DG_DEV_TIMEOUT);
}

// Apply the epilogue to 32 consecutive accumulator columns [col0, col0 + 32) of one row.
// `g` holds gate values for EPI_GELU_GATEUP (then `v` holds the matching up values).
DG_DEVINL void epi_store(const GemmArgs& a, int epi, int m, int n_tile, int row, int col_in_tile, int BNv,
                         const float (&v)[32], const float* g) {
    if (epi == EPI_F32) {
        const int64_t r = (int64_t)m * BM + row;
        if (r >= a.m_valid) return;
        const int c0 = n_tile * BNv + col_in_tile;
        float* o = static_cast<float*>(a.out) + r * a.ldo + c0;
        if (c0 + 32 <= a.n_valid && ((reinterpret_cast<uintptr_t>(o) & 15u) == 0)) {
#pragma unroll
            for (int i = 0; i < 32; i += 4) *reinterpret_cast<float4*>(o + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        } else {
            for (int i = 0; i < 32; ++i)
                if (c0 + i < a.n_valid) o[i] = v[i];
        }
        return;
    }
    uint32_t pk[16];
    int c0;
    int64_t r;
    uint16_t* base;
    if (epi == EPI_GELU_GATEUP) {
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(gelu_tanh(g[2 * i]) * v[2 * i], gelu_tanh(g[2 * i + 1]) * v[2 * i + 1]);
        c0 = n_tile * (BNv / 2) + col_in_tile;
        r = (int64_t)m * BM + row;
        base = static_cast<uint16_t*>(a.out);
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
        c0 = n_tile * BNv + col_in_tile;
        if (epi == EPI_SCATTER_BF16) {
            const int pos = (m % a.tpc) * BM + row;
            if (pos >= a.L) return;
            r = (int64_t)canvas_of(a, m) * a.L + pos;
        } else {
            r = (int64_t)m * BM + row;
        }
        base = static_cast<uint16_t*>(a.out);
    }
    uint16_t* o = base + r * a.ldo + c0;
    if (c0 + 32 <= a.n_valid && ((reinterpret_cast<uintptr_t>(o) & 15u) == 0)) {
#pragma unroll
        for (int i = 0; i < 16; i += 4) *reinterpret_cast<uint4*>(o + 2 * i) = make_uint4(pk[i], pk[i + 1], pk[i + 2], pk[i + 3]);
    } else {
        for (int i = 0; i < 32; ++i)
            if (c0 + i < a.n_valid) o[i] = (uint16_t)((i & 1) ? (pk[i >> 1] >> 16) : (pk[i >> 1] & 0xFFFFu));
    }
}

// ------------------------------------------------------------------ LM-head epilogue
// EPI_LOGIT_STATS: one row's part of the logits over one tile of BN columns.  The fp32
// accumulator is rounded to bf16 (the stored logits: 16-byte stores into the caller's
// [n][L][ld] rows), and the softmax state of exactly those stored values is recorded for the
// row: the maximum m, the count c of entries equal to it, r = sum over the others of
// 2^((x - m) k2), t = sum of 2^((x - m) k2) (x - m) k2 (k2 = log2(e) / T), and the first
// column holding m.  -inf entries are left out of the state; a NaN or +inf marks the record
// (c = NaN).  The records of a row merge in any order to the row's statistics.
constexpr float kStatsMinExponent = -256.f;  // 2^-256 is 0 in fp32: keeps t finite

template <int BN>
DG_DEVINL void logit_stats_tile(const GemmArgs& a, int m, int n_tile, int row, uint32_t tbase) {
    const int pos = (m % a.tpc) * BM + row;
    const bool live = pos < a.L;  // the canvas's last tile may hold padding rows
    const int cz = canvas_of(a, m);
    const int64_t r = (int64_t)cz * a.L + pos;
    const float k2 = kLog2e / a.params[cz].temperature;
    uint16_t* orow = static_cast<uint16_t*>(a.out) + r * a.ldo;
    float M = -INFINITY, cnt = 0.f, rs = 0.f, ts = 0.f;
    int idx = 0x7fffffff;
    bool bad = false;
#pragma unroll 1
    for (int ch = 0; ch < BN / 32; ++ch) {
        float v[32];
        dg::tmem_ld32(tbase + ch * 32, v);  // whole warp
        const int c0 = n_tile * BN + ch * 32;
        if (!live || c0 >= a.n_valid) continue;
        const int nv = min(32, a.n_valid - c0);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
        uint16_t* o = orow + c0;
        if (nv == 32) {
#pragma unroll
            for (int i = 0; i < 16; i += 4) *reinterpret_cast<uint4*>(o + 2 * i) = make_uint4(pk[i], pk[i + 1], pk[i + 2], pk[i + 3]);
        } else {
            for (int i = 0; i < nv; ++i) o[i] = (uint16_t)((i & 1) ? (pk[i >> 1] >> 16) : (pk[i >> 1] & 0xFFFFu));
        }
        float x[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            x[2 * i] = __uint_as_float(pk[i] << 16);
            x[2 * i + 1] = __uint_as_float(pk[i] & 0xffff0000u);
        }
        float cm = -INFINITY;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (j < nv) {
                bad |= (x[j] != x[j]) || (x[j] == INFINITY);
                cm = fmaxf(cm, x[j]);
            }
        }
        if (cm > M) {  // a new maximum: the entries so far move below it
            if (cnt > 0.f || rs > 0.f) {
                const float d = (M - cm) * k2, al = ex2(d), sum = cnt + rs;
                ts = al * (ts + d * sum);
                rs = al * sum;
                cnt = 0.f;
            }
            M = cm;
            idx = 0x7fffffff;
        }
        if (cm == -INFINITY) continue;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            if (j < nv && x[j] > -INFINITY) {
                if (x[j] == M) {
                    cnt += 1.f;
                    idx = min(idx, c0 + j);
                } else if (x[j] == x[j]) {
                    const float d = fmaxf((x[j] - M) * k2, kStatsMinExponent);
                    const float e = ex2(d);
                    rs += e;
                    ts = fmaf(e, d, ts);
                }
            }
        }
    }
    if (live) {
        const int64_t R = a.stats_rows;
        float* st = a.stats + (int64_t)n_tile * 5 * R + r;
        st[0] = M;
        st[R] = bad ? __int_as_float(0x7fc00000) : cnt;
        st[2 * R] = rs;
        st[3 * R] = ts;
        st[4 * R] = __int_as_float(idx);
    }
}

// ------------------------------------------------------------------ the GEMM kernel
// Launched as clusters of cm CTAs: cm = 2 for the CTA-pair configurations (cta_group::2
// MMAs over the pair's 256 rows), cm = 1 otherwise.  Every CTA loads its own operand tiles
// with plain TMA copies; CTAs that share a tile find it in L2.
template <class C>
__global__ void __launch_bounds__(C::kThreads, 1)
    k_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
           const __grid_constant__ CUtensorMap tmB1, const GemmArgs a) {
    extern __shared__ __align__(1024) unsigned char g_smem_raw[];
    // 1024-byte aligned stage ring after the barrier block
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(g_smem_raw) + 1023) & ~uintptr_t(1023));
    GemmShared& sh = *reinterpret_cast<GemmShared*>(smem + (size_t)C::STAGES * C::kStageBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    cg::cluster_group cluster = cg::this_cluster();
    const int cm = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();
    const int64_t cid = blockIdx.x / cm, ncl = gridDim.x / cm;
    const uint16_t mask = (uint16_t)((1u << cm) - 1u);
    constexpr bool PAIR = C::kPair;
    const bool leader = !PAIR || rank == 0;  // the pair's MMAs are issued by its first CTA

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            dg::mbar_init(&sh.full[s], 1);
            // pair: one arrival per transform warp of the stage's group in both CTAs, in the
            // first CTA's barrier
            // (without a transform: the second CTA's relay, once its own stage has landed)
            dg::mbar_init(&sh.xform[s], PAIR ? (C::kXform ? 2 * (C::kXformWarps / DG_XFORM_GROUPS) : 1)
                                              : (C::kXform ? C::kXformThreads / DG_XFORM_GROUPS : 1));
            dg::mbar_init(&sh.empty[s], 1);  // released by the (pair's) MMA commit
        }
        for (int i = 0; i < C::kNAcc; ++i) {
            dg::mbar_init(&sh.accf[i], 1);
            dg::mbar_init(&sh.acce[i], PAIR ? 2 * 4 : 128);  // pair: one per epilogue warp of both CTAs
        }
        sh.abort_flag = 0;
        dg::fence_mbar_init();
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            dg::tmem_alloc_pair(&sh.tmem_base, C::kTmemCols);
            dg::tmem_relinquish_pair();
        } else {
            dg::tmem_alloc(&sh.tmem_base, C::kTmemCols);
            dg::tmem_relinquish();
        }
    }
    dg::tc_fence_before();
    cluster.sync();  // the peer's barriers are initialised before any pair commit or arrival lands
    dg::tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    // the prologue above overlaps the previous kernel; its outputs (plan, lse, A, B) are read below
    dg::pdl_wait();
    dg::pdl_release();
    const int mt = active_m_tiles(a);
    if (threadIdx.x == 0) sh.splits = active_splits(a, mt);  // once per CTA, shared
    __syncthreads();
    const int splits = sh.splits;
    const int64_t n_groups = mt > 0 ? group_count(a, mt, cm, splits) : 0;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            dg::prefetch_tmap(&tmA);
            dg::prefetch_tmap(&tmB0);
            if (C::kBMode == B_KMAJOR_GATEUP) dg::prefetch_tmap(&tmB1);
            uint32_t it = 0;
            const bool pace = DG_PE_PACE && C::kXform && a.pace != nullptr;
            unsigned item_no = 0;
            for (int64_t G = cid; G < n_groups && !aborted(sh); G += ncl, ++item_no) {
                const Item im = decode(a, mt, cm, rank, G, splits);
                if (pace && item_no > 0) pace_wait(a.pace, item_no * gridDim.x, a.status);
                int cz = 0, crow = 0;
                if (C::kXform || C::kAMode == A_TMA_CANVAS) {
                    cz = canvas_of(a, im.m_load);
                    crow = (im.m_load % a.tpc) * BM;
                }
                for (int kb = im.kb_lo; kb < im.kb_hi; ++kb, ++it) {
                    const int s = (int)(it % C::STAGES);
                    const uint32_t ph = (it / C::STAGES) & 1u;
                    if (!dg::mbar_wait(&sh.empty[s], ph ^ 1u)) { do_abort(sh, a.status); break; }
                    unsigned char* st = smem + (size_t)s * C::kStageBytes;
                    unsigned char* sA = st;
                    unsigned char* sB = st + C::kATileBytes;
                    unsigned char* sF = st + C::kATileBytes + C::kBTileBytes;  // fp32 staging
                    dg::mbar_arrive_expect_tx(&sh.full[s], C::kTxBytes);
                    const int k0 = kb * C::BK;
                    if (C::kAMode == A_TMA) {
                        dg::tma_load_2d(sA, &tmA, k0, im.m_load * BM, &sh.full[s]);
                    } else if (C::kAMode == A_SOFTMAX_BF16 || C::kAMode == A_TMA_CANVAS) {
                        dg::tma_load_3d(sA, &tmA, k0, crow, cz, &sh.full[s]);
                    } else {
                        // fp32 logits: BK = 32 columns = one 128-byte swizzle row per tile row
                        dg::tma_load_3d(sF, &tmA, k0, crow, cz, &sh.full[s]);
                    }
                    if (C::kBMode == B_MNMAJOR) {
                        // [K][N] embedding rows: one 64-column (128-byte) atom column per load
                        if (PAIR) {
                            // this CTA's half of each 256-column slab h: atoms 2h, 2h + 1
#pragma unroll
                            for (int h = 0; h < C::BN / 256; ++h)
#pragma unroll
                                for (int at = 0; at < 2; ++at)
                                    dg::tma_load_2d(sB + (2 * h + at) * (C::BK * 128), &tmB0,
                                                    im.n * C::BN + h * 256 + rank * 128 + at * 64, k0, &sh.full[s]);
                        } else {
#pragma unroll
                            for (int j = 0; j < C::BN / 64; ++j)
                                dg::tma_load_2d(sB + j * (C::BK * 128), &tmB0, im.n * C::BN + j * 64, k0, &sh.full[s]);
                        }
                    } else if (C::kBMode == B_KMAJOR) {
                        // pair: this CTA's half of the tile's rows (box of BN / 2 rows)
                        dg::tma_load_2d(sB, &tmB0, k0, im.n * C::BN + (PAIR ? rank * (C::BN / 2) : 0), &sh.full[s]);
                    } else if (PAIR) {
                        // gate rows from the first CTA, up rows from the second
                        dg::tma_load_2d(sB, rank == 0 ? &tmB0 : &tmB1, k0, im.n * (C::BN / 2), &sh.full[s]);
                    } else {
                        // gate rows in the first half of the tile, up rows in the second
                        dg::tma_load_2d(sB, &tmB0, k0, im.n * (C::BN / 2), &sh.full[s]);
                        dg::tma_load_2d(sB + (C::BN / 2) * C::BK * 2, &tmB1, k0, im.n * (C::BN / 2), &sh.full[s]);
                    }
                }
                if (pace) atomicAdd(a.pace, 1u);
            }
            // never leave with a copy still landing in this CTA's shared memory
            if (aborted(sh)) {
                for (int s = 0; s < C::STAGES; ++s) (void)dg::mbar_wait(&sh.full[s], 0);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (relay in the pair's second CTA)
        if (PAIR && !C::kXform && lane == 0 && !leader) {
            // tell the first CTA when this CTA's part of each stage has landed
            uint32_t it = 0;
            bool ok = true;
            for (int64_t G = cid; G < n_groups && ok && !aborted(sh); G += ncl) {
                const Item im = decode(a, mt, cm, rank, G, splits);
                for (int kb = im.kb_lo; kb < im.kb_hi; ++kb, ++it) {
                    const int s = (int)(it % C::STAGES);
                    if (!dg::mbar_wait(&sh.full[s], (it / C::STAGES) & 1u)) { ok = false; break; }
                    dg::mbar_arrive_remote(dg::mapa_shared(&sh.xform[s], 0));
                }
            }
            if (!ok) do_abort(sh, a.status);
        }
        if (lane == 0 && leader) {
            constexpr uint32_t idesc_pair = instr_desc(2 * BM, 256, C::kBMode == B_MNMAJOR);
            constexpr uint32_t idesc_mn = instr_desc(BM, C::BN > 256 ? 256 : C::BN, true);
            constexpr uint32_t idesc_k = instr_desc(BM, C::BN > 256 ? 256 : C::BN, false);
            constexpr uint32_t idesc = (C::kBMode == B_MNMAJOR) ? idesc_mn : idesc_k;
            uint32_t it = 0, acc_it = 0;
            for (int64_t G = cid; G < n_groups && !aborted(sh); G += ncl, ++acc_it) {
                const Item im = decode(a, mt, cm, rank, G, splits);
                const int ab = (int)(acc_it % C::kNAcc);
                const uint32_t aph = (acc_it / C::kNAcc) & 1u;
                if (!dg::mbar_wait(&sh.acce[ab], aph ^ 1u)) {
                    do_abort(sh, a.status);
                    break;
                }
                dg::tc_fence_after();
                const uint32_t dacc = tmem + (uint32_t)(ab * C::kAccCols);
                bool ok = true;
                for (int kb = im.kb_lo; kb < im.kb_hi; ++kb, ++it) {
                    const int s = (int)(it % C::STAGES);
                    const uint32_t ph = (it / C::STAGES) & 1u;
                    // pair: the transform warps of both CTAs report (after their own full waits);
                    // without a transform, this CTA's stage and the second CTA's relay
                    if ((!PAIR || !C::kXform) && !dg::mbar_wait(&sh.full[s], ph)) { ok = false; break; }
                    if (PAIR && !dg::mbar_wait(&sh.xform[s], ph)) { ok = false; break; }
                    if (!PAIR && C::kXform && !dg::mbar_wait(&sh.xform[s], ph)) { ok = false; break; }
                    dg::tc_fence_after();
                    const uint32_t sA = dg::smem_u32(smem + (size_t)s * C::kStageBytes);
                    const uint32_t sB = sA + C::kATileBytes;
#pragma unroll
                    for (int kk = 0; kk < C::BK / 16; ++kk) {
                        const uint64_t ad = smem_desc(sA + kk * 32, 16, 8 * C::BK * 2, C::kASwizzle);
                        const uint32_t accum = (kb > im.kb_lo || kk > 0) ? 1u : 0u;
                        if constexpr (PAIR && C::kBMode == B_MNMAJOR) {
                            // two N = 256 slabs; this CTA's B holds 2 atom columns of each
#pragma unroll
                            for (int h = 0; h < C::BN / 256; ++h) {
                                const uint64_t bd = smem_desc(sB + h * 2 * (C::BK * 128) + kk * 16 * 128, C::BK * 128, 1024, 128);
                                dg::tc_mma_f16_pair(dacc + h * 256, ad, bd, idesc_pair, accum);
                            }
                        } else if constexpr (PAIR) {
                            // K-major B: this CTA's BN / 2 rows
                            const uint64_t bd = smem_desc(sB + kk * 32, 16, 8 * C::BK * 2, C::kASwizzle);
                            dg::tc_mma_f16_pair(dacc, ad, bd, idesc_pair, accum);
                        } else if (C::kBMode == B_MNMAJOR) {
                            // N-major B: LBO = distance between 64-column atom columns, SBO = 8 K rows
#pragma unroll
                            for (int h = 0; h < C::BN / 256; ++h) {
                                const uint64_t bd = smem_desc(sB + h * 4 * (C::BK * 128) + kk * 16 * 128, C::BK * 128, 1024, 128);
                                dg::tc_mma_f16(dacc + h * 256, ad, bd, idesc, accum);
                            }
                        } else {
                            const uint64_t bd = smem_desc(sB + kk * 32, 16, 8 * C::BK * 2, C::kASwizzle);
                            dg::tc_mma_f16(dacc, ad, bd, idesc, accum);
                        }
                    }
                    // frees the stage (in both CTAs of a pair) once these MMAs have read it
                    if constexpr (PAIR) dg::tc_commit_pair_mc(&sh.empty[s], mask);
                    else dg::tc_commit(&sh.empty[s]);
                }
                if (!ok) { do_abort(sh, a.status); break; }
                if constexpr (PAIR) dg::tc_commit_pair_mc(&sh.accf[ab], mask);  // both CTAs' accumulators complete
                else dg::tc_commit(&sh.accf[ab]);                              // accumulator complete
            }
        }
    } else if (warp < 6) {
        // ------------------------------------------------ epilogue (warps 2..5)
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        uint32_t acc_it = 0;
        for (int64_t G = cid; G < n_groups && !aborted_warp(sh); G += ncl, ++acc_it) {
            const Item im = decode(a, mt, cm, rank, G, splits);
            const int ab = (int)(acc_it % C::kNAcc);
            const uint32_t aph = (acc_it / C::kNAcc) & 1u;
            if (!dg::mbar_wait_warp(&sh.accf[ab], aph, 256)) { do_abort(sh, a.status); break; }
            dg::tc_fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(ab * C::kAccCols);
            if (!im.valid) {
                // padding member of the group: nothing to store
            } else if (splits > 1) {
                // partial tile in column-quad order [BN / 4][BM][4]: the warp's 32 rows store
                // 512 contiguous bytes per instruction instead of 16 bytes in each of 32 rows
                float* dst = a.partial + (size_t)im.w * (BM * C::BN) + (size_t)row * 4;
                for (int ch = 0; ch < C::BN / 32; ++ch) {
                    float v[32];
                    dg::tmem_ld32(tbase + ch * 32, v);
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4*>(dst + (size_t)((ch * 32 + i) / 4) * (BM * 4)) =
                            make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                }
            } else if (a.epi == EPI_LOGIT_STATS) {
                logit_stats_tile<C::BN>(a, im.m, im.n, row, tbase);
            } else if (a.epi == EPI_GELU_GATEUP) {
                for (int ch = 0; ch < C::BN / 64; ++ch) {
                    float g[32], u[32];
                    dg::tmem_ld32(tbase + ch * 32, g);
                    dg::tmem_ld32(tbase + C::BN / 2 + ch * 32, u);
                    epi_store(a, a.epi, im.m, im.n, row, ch * 32, C::BN, u, g);
                }
            } else {
                for (int ch = 0; ch < C::BN / 32; ++ch) {
                    float v[32];
                    dg::tmem_ld32(tbase + ch * 32, v);
                    epi_store(a, a.epi, im.m, im.n, row, ch * 32, C::BN, v, nullptr);
                }
            }
            dg::tc_fence_before();
            if (PAIR) {
                __syncwarp();
                if (lane == 0) dg::mbar_arrive_remote(dg::mapa_shared(&sh.acce[ab], 0));
            } else {
                dg::mbar_arrive(&sh.acce[ab]);
            }
        }
    } else {
        // ------------------------------------------------ softmax transform (warps 6..13)
        if (C::kXform) {
            // kXG groups of transform threads take the stages in turn (stage it goes to group
            // it % kXG), so each group has kXG stages' worth of MMA time for one stage's chain
            // (barrier wait, shared loads, exponentials, stores, proxy fence, arrival); a
            // thread converts kRows whole tile rows of its group's stages
            constexpr int kXG = DG_XFORM_GROUPS;
            constexpr int kGT = C::kXformThreads / kXG;       // threads per group
            constexpr int kRows = BM / kGT;                    // tile rows per thread
            static_assert(kGT >= 32 && kGT <= BM && BM % kGT == 0, "whole warps, whole rows per group");
            const int xt = threadIdx.x - 192;
            const int grp = xt / kGT;
            const int t0 = xt % kGT;
            uint32_t it = 0;
            for (int64_t G = cid; G < n_groups && !aborted_warp(sh); G += ncl) {
                const Item im = decode(a, mt, cm, rank, G, splits);
                const int cz = canvas_of(a, im.m_load);
                const dg_canvas_params pr = a.params[cz];
                const float kx = kLog2e / pr.temperature;
                float lbs[kRows];
#pragma unroll
                for (int r = 0; r < kRows; ++r) {
                    const int pos = (im.m_load % a.tpc) * BM + t0 + r * kGT;
                    lbs[r] = (pos < a.L) ? a.lse[(int64_t)cz * a.L + pos] * kLog2e : 0.f;
                }
                bool ok = true;
                for (int kb = im.kb_lo; kb < im.kb_hi; ++kb, ++it) {
                    if ((int)(it % kXG) != grp) continue;
                    const int s = (int)(it % C::STAGES);
                    const uint32_t ph = (it / C::STAGES) & 1u;
                    // every lane polls; the outcome is made warp-uniform (the warp arrives as one)
                    if (!__all_sync(0xffffffffu, dg::mbar_wait(&sh.full[s], ph))) { ok = false; break; }
                    unsigned char* st = smem + (size_t)s * C::kStageBytes;
                    const int64_t kbase = (int64_t)kb * C::BK;
                    const bool tail = kbase + C::BK > a.K;
#pragma unroll
                    for (int r = 0; r < kRows; ++r) {
                        const int t = t0 + r * kGT;
                        const float lb = lbs[r];
                        unsigned char* rowA = st + t * (C::BK * 2);
                        // one tile row = BK bf16 = BK/8 16-byte chunks; the swizzle permutes chunks
                        // within the row, so chunk c of the row sits at c ^ ((t >> sh) & mask)
                        constexpr int kChunks = C::BK / 8;
                        const int sw = (C::kASwizzle == 128) ? (t & 7) : ((t >> 1) & 3);
#pragma unroll
                        for (int cc = 0; cc < kChunks; ++cc) {
                            const int c = cc;
                            const int pc = c ^ sw;
                            float x[8];
                            if (C::kAMode == A_SOFTMAX_BF16) {
                                const uint4 qv = *reinterpret_cast<const uint4*>(rowA + pc * 16);
                                x[0] = __uint_as_float(qv.x << 16); x[1] = __uint_as_float(qv.x & 0xffff0000u);
                                x[2] = __uint_as_float(qv.y << 16); x[3] = __uint_as_float(qv.y & 0xffff0000u);
                                x[4] = __uint_as_float(qv.z << 16); x[5] = __uint_as_float(qv.z & 0xffff0000u);
                                x[6] = __uint_as_float(qv.w << 16); x[7] = __uint_as_float(qv.w & 0xffff0000u);
                            } else {
                                // fp32 staging row: 32 floats = 128 bytes, 128-byte swizzle
                                const unsigned char* rowF = st + C::kATileBytes + C::kBTileBytes + t * 128;
                                const float4 f0 = *reinterpret_cast<const float4*>(rowF + (((2 * c) ^ (t & 7)) * 16));
                                const float4 f1 = *reinterpret_cast<const float4*>(rowF + (((2 * c + 1) ^ (t & 7)) * 16));
                                x[0] = f0.x; x[1] = f0.y; x[2] = f0.z; x[3] = f0.w;
                                x[4] = f1.x; x[5] = f1.y; x[6] = f1.z; x[7] = f1.w;
                            }
                            // exponent arguments two at a time (fma.rn.f32x2: the same single
                            // rounding per element as fmaf)
                            float pz[8];
                            {
                                uint64_t kk, bb;
                                asm("mov.b64 %0, {%1, %1};" : "=l"(kk) : "f"(kx));
                                asm("mov.b64 %0, {%1, %1};" : "=l"(bb) : "f"(-lb));
#pragma unroll
                                for (int j = 0; j < 8; j += 2) {
                                    uint64_t xx, rr;
                                    asm("mov.b64 %0, {%1, %2};" : "=l"(xx) : "f"(x[j]), "f"(x[j + 1]));
                                    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rr) : "l"(xx), "l"(kk), "l"(bb));
                                    float lo, hi;
                                    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(rr));
                                    pz[j] = ex2(lo);
                                    pz[j + 1] = ex2(hi);
                                }
                            }
                            if (tail) {
#pragma unroll
                                for (int j = 0; j < 8; ++j)
                                    if (kbase + c * 8 + j >= a.K) pz[j] = 0.f;
                            }
                            *reinterpret_cast<uint4*>(rowA + pc * 16) =
                                make_uint4(pack_bf16x2(pz[0], pz[1]), pack_bf16x2(pz[2], pz[3]),
                                           pack_bf16x2(pz[4], pz[5]), pack_bf16x2(pz[6], pz[7]));
                        }
                    }  // rows
                    dg::fence_proxy_async_smem();  // make the generic-proxy writes visible to tcgen05
                    if (PAIR) {
                        __syncwarp();
                        if (lane == 0) dg::mbar_arrive_remote(dg::mapa_shared(&sh.xform[s], 0));
                    } else {
                        dg::mbar_arrive(&sh.xform[s]);
                    }
                }
                if (!ok) { do_abort(sh, a.status); break; }
            }
        }
    }

    dg::tc_fence_before();
    // no CTA of a pair leaves while its peer may still signal its barriers
    cluster.sync();
    if (warp == 1) {
        dg::tc_fence_after();
        if constexpr (PAIR) dg::tmem_dealloc_pair(tmem, C::kTmemCols);
        else dg::tmem_dealloc(tmem, C::kTmemCols);
    }
}

// ------------------------------------------------------------------ split-K fix-up
// Adds the k-slice partials of each tile in slice order and applies the epilogue.  Every
// thread owns 4 consecutive output columns of a row; consecutive threads take consecutive
// rows of one column quad, which are adjacent in the partial tiles' [BN / 4][BM][4] order
// (float4 loads, coalesced across the warp), and the tiles are spread over gridDim.y CTAs
// each.  For the gate/up epilogue the output columns are the tile's first BN/2 (gate)
// columns, each paired with the up column BN/2 later.
template <int BN, bool GU>
__global__ void __launch_bounds__(256, GU ? 1 : 4) k_fixup(const GemmArgs a) {
    dg::pdl_wait();
    dg::pdl_release();
    const int mt = active_m_tiles(a);
    __shared__ int splits_sh;
    if (threadIdx.x == 0) splits_sh = active_splits(a, mt);  // once per CTA, shared
    __syncthreads();
    const int splits = splits_sh;
    if (splits <= 1) return;  // the device's plan did not split K: nothing to add
    const int64_t T = (int64_t)mt * a.n_tiles;
    const int64_t t = blockIdx.x;
    if (t >= T) return;
    const int n = (int)((uint32_t)t / (uint32_t)mt), m = (int)((uint32_t)t - (uint32_t)n * (uint32_t)mt);
    constexpr bool gu = GU;  // a.epi == EPI_GELU_GATEUP
    const int out_cols = gu ? BN / 2 : BN;
    const int quads = BM * out_cols / 4;
    const int per_cta = (quads + gridDim.y - 1) / gridDim.y;
    const int q0 = blockIdx.y * per_cta, q1 = min(quads, q0 + per_cta);
    for (int qd = q0 + threadIdx.x; qd < q1; qd += blockDim.x) {
        const int row = qd % BM;
        const int cq = qd / BM;  // column quad
        const int col = cq * 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f), up = make_float4(0.f, 0.f, 0.f, 0.f);
        // kU slices' loads in flight at once, added in slice order (read once: streaming loads)
        constexpr int kU = 8;
        for (int s0 = 0; s0 < splits; s0 += kU) {
            float4 v[kU], u[kU];
#pragma unroll
            for (int j = 0; j < kU; ++j) {
                if (s0 + j >= splits) continue;
                const float* src = a.partial + (size_t)((s0 + j) * T + t) * (BM * BN) + ((size_t)cq * BM + row) * 4;
                v[j] = __ldcs(reinterpret_cast<const float4*>(src));
                if (gu) u[j] = __ldcs(reinterpret_cast<const float4*>(src + (size_t)(BN / 8) * BM * 4));
            }
#pragma unroll
            for (int j = 0; j < kU; ++j) {
                if (s0 + j >= splits) continue;
                acc.x += v[j].x;
                acc.y += v[j].y;
                acc.z += v[j].z;
                acc.w += v[j].w;
                if (gu) {
                    up.x += u[j].x;
                    up.y += u[j].y;
                    up.z += u[j].z;
                    up.w += u[j].w;
                }
            }
        }
        int64_t r;
        int c0;
        if (a.epi == EPI_SCATTER_BF16) {
            const int pos = (m % a.tpc) * BM + row;
            if (pos >= a.L) continue;
            r = (int64_t)canvas_of(a, m) * a.L + pos;
            c0 = n * BN + col;
        } else {
            r = (int64_t)m * BM + row;
            c0 = n * out_cols + col;
        }
        if (a.epi == EPI_F32) {
            if (r >= a.m_valid) continue;
            float* o = static_cast<float*>(a.out) + r * a.ldo + c0;
            const float vv[4] = {acc.x, acc.y, acc.z, acc.w};
            for (int i = 0; i < 4; ++i)
                if (c0 + i < a.n_valid) o[i] = vv[i];
            continue;
        }
        if (gu) {
            acc.x = gelu_tanh(acc.x) * up.x;
            acc.y = gelu_tanh(acc.y) * up.y;
            acc.z = gelu_tanh(acc.z) * up.z;
            acc.w = gelu_tanh(acc.w) * up.w;
        }
        uint16_t* o = static_cast<uint16_t*>(a.out) + r * a.ldo + c0;
        const uint32_t p0 = pack_bf16x2(acc.x, acc.y), p1 = pack_bf16x2(acc.z, acc.w);
        if (c0 + 4 <= a.n_valid && ((reinterpret_cast<uintptr_t>(o) & 7u) == 0)) {
            *reinterpret_cast<uint2*>(o) = make_uint2(p0, p1);
        } else {
            const uint16_t hv[4] = {(uint16_t)(p0 & 0xFFFFu), (uint16_t)(p0 >> 16), (uint16_t)(p1 & 0xFFFFu),
                                    (uint16_t)(p1 >> 16)};
            for (int i = 0; i < 4; ++i)
                if (c0 + i < a.n_valid) o[i] = hv[i];
        }
    }
}

// ------------------------------------------------------------------ self-conditioning helpers
DG_DEVINL bool self_cond_on(const dg_canvas_params& p, const uint8_t* converged, int64_t c) {
    return (p.flags & DG_ACTIVE) && (p.flags & DG_SELF_COND) && !(p.flags & DG_READ_ONLY) &&
           !(converged && converged[c]) && p.temperature > 0.f;
}

// Compact list of canvases in original order: those whose feedback is computed this step
// (mode 0) or the active ones (mode 1, the LM head's rows).  Per chunk of blockDim.x
// canvases, warp ballots, an exclusive prefix over the warps' counts.
// Called by every thread of one block.
DG_DEVINL void plan_list(const dg_canvas_params* __restrict__ params, const uint8_t* __restrict__ converged,
                         int64_t n, int32_t* __restrict__ plan, int mode) {
    __shared__ int warp_base[32];
    __shared__ int total;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    int count = 0;  // canvases listed before this chunk (same in every thread)
    for (int64_t base = 0; base < n; base += blockDim.x) {
        const int64_t c = base + threadIdx.x;
        const bool on = c < n && (mode == 0 ? self_cond_on(params[c], converged, c)
                                            : (params[c].flags & DG_ACTIVE) != 0u);
        const unsigned ballot = __ballot_sync(0xffffffffu, on);
        if (lane == 0) warp_base[warp] = __popc(ballot);
        __syncthreads();
        if (warp == 0) {
            const int v = lane < nwarps ? warp_base[lane] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (lane < nwarps) warp_base[lane] = incl - v;
            if (lane == 31) total = incl;
        }
        __syncthreads();
        if (on) plan[1 + count + warp_base[warp] + __popc(ballot & ((1u << lane) - 1u))] = (int32_t)c;
        count += total;
        __syncthreads();  // warp_base and total are rewritten by the next chunk
    }
    if (threadIdx.x == 0) plan[0] = count;
}

__global__ void k_plan(const dg_canvas_params* __restrict__ params, const uint8_t* __restrict__ converged,
                       int64_t n, int32_t* __restrict__ plan, int mode) {
    dg::pdl_wait();
    dg::pdl_release();
    plan_list(params, converged, n, plan, mode);
}

// The feedback plan (block (0, 0), as k_plan mode 0; it also zeroes P.E's pacing counter) and
// the zeroing of the feedback rows of canvases that get none this step: grid (CTAs per canvas,
// canvases), 16-byte stores (d is a multiple of 8 and delta_emb 16-byte aligned).
__global__ void k_zero_rows(const dg_canvas_params* __restrict__ params, const uint8_t* __restrict__ converged,
                            int64_t n, int32_t L, int32_t d, uint16_t* __restrict__ delta,
                            int32_t* __restrict__ plan, unsigned* __restrict__ pace) {
    dg::pdl_wait();
    dg::pdl_release();
    if (blockIdx.x == 0 && blockIdx.y == 0) {
        if (threadIdx.x == 0) *pace = 0u;
        plan_list(params, converged, n, plan, 0);
    }
    const int64_t c = blockIdx.y;
    if (self_cond_on(params[c], converged, c)) return;
    const int64_t vecs = (int64_t)L * d / 8;
    uint4* row = reinterpret_cast<uint4*>(delta + c * (int64_t)L * d);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < vecs; i += (int64_t)gridDim.x * blockDim.x)
        row[i] = make_uint4(0u, 0u, 0u, 0u);
}

// The feedback rows of canvases that got feedback although they converged this step (the
// feedback was computed before the convergence was known): zeroed, as if planned without
// them.  Grid (CTAs per canvas, canvases).
__global__ void k_zero_converged(const dg_canvas_params* __restrict__ params, const uint8_t* __restrict__ converged,
                                 int32_t L, int32_t d, uint16_t* __restrict__ delta) {
    dg::pdl_wait();
    dg::pdl_release();
    const int64_t c = blockIdx.y;
    if (!self_cond_on(params[c], nullptr, c) || !converged[c]) return;
    const int64_t vecs = (int64_t)L * d / 8;
    uint4* row = reinterpret_cast<uint4*>(delta + c * (int64_t)L * d);
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < vecs; i += (int64_t)gridDim.x * blockDim.x)
        row[i] = make_uint4(0u, 0u, 0u, 0u);
}

// ------------------------------------------------------------------ host side
// Pipeline depths (shared-memory stages) of the self-conditioning GEMMs.
#ifndef DG_PE_STAGES
#define DG_PE_STAGES 8
#endif
#ifndef DG_MLP_STAGES
#define DG_MLP_STAGES 6
#endif
using PEbf16 = Cfg<A_SOFTMAX_BF16, B_MNMAJOR, 512, 32, DG_PE_STAGES, true>;
using PEfp32 = Cfg<A_SOFTMAX_FP32, B_MNMAJOR, 512, 32, 5, true>;
using PEprob = Cfg<A_TMA, B_MNMAJOR, 512, 32, DG_PE_STAGES, true>;  // plain N-major B: CTA pairs
using GateUp = Cfg<A_TMA, B_KMAJOR_GATEUP, 256, 64, DG_MLP_STAGES, true>;
using Down = Cfg<A_TMA, B_KMAJOR, 256, 64, DG_MLP_STAGES, true>;
using DownSingle = Cfg<A_TMA, B_KMAJOR, 256, 64, 4>;  // plain GEMMs (K-major B) on one CTA per tile
// LM head: hidden rows of the listed canvases (3D map) times W_lm [V][d] (K-major), CTA pairs
using LmHead = Cfg<A_TMA_CANVAS, B_KMAJOR, 256, 64, DG_MLP_STAGES, true>;

constexpr size_t align256(size_t x) { return (x + 255) / 256 * 256; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct LaunchPlan {
    int cm;        // CTAs per cluster
    int clusters;  // concurrent clusters (persistent grid = clusters * cm CTAs)
    int splits;    // k-slices (for the host's m-tile count)
    int min_slice;
    int64_t max_slots;
    int split_below;  // percent
};

// Cluster size, persistent grid and k-slices for a GEMM.  Pair configurations run as 2-CTA
// clusters (as many as fit at once), the others one CTA per cluster on every SM.  The
// k-slices are then chosen for the number of clusters, within `max_slots` partial tiles,
// with slices of at least `min_slice` k-blocks, and only when the unsplit work would fill
// less than `split_below` of the clusters' last round.
template <class C>
bool plan_gemm(const GemmArgs& a, int64_t max_slots, LaunchPlan* pl, int min_slice = 256, int split_below = 101) {
    auto kern = k_gemm<C>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem) != cudaSuccess)
        return false;
    const int P = dghost::sm_count();
    if (P <= 0) return false;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int cm = C::kPair ? 2 : 1;
    int clusters = P;
    if (C::kPair) {
        attr[0].val.clusterDim.x = 2u;
        cfg.gridDim = dim3((unsigned)((P / 2) * 2), 1, 1);
        int nc = 0;
        if (cudaOccupancyMaxActiveClusters(&nc, kern, &cfg) != cudaSuccess || nc <= 0)
            return false;  // a pair kernel runs only as 2-CTA clusters
        clusters = nc;
    }
    const int64_t per_split = (int64_t)a.n_tiles * ((a.m_tiles + cm - 1) / cm);
    const int splits = plan_splits(per_split, a.m_tiles, a.n_tiles, a.k_blocks, clusters, min_slice, max_slots,
                                   split_below);
    pl->min_slice = min_slice;
    pl->max_slots = max_slots;
    pl->split_below = split_below;
    pl->cm = cm;
    pl->clusters = clusters;
    pl->splits = splits;
    return true;
}

template <class C>
dg_status launch_gemm(const void* tmA, const void* tmB0, const void* tmB1, const GemmArgs& a, const LaunchPlan& pl,
                      cudaStream_t stream) {
    auto kern = k_gemm<C>;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)pl.cm;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // the kernel waits after its prologue
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    // with the k-slices chosen on the device the work may exceed the host's count: the full
    // persistent grid (CTAs without work leave after their prologue)
    const int64_t groups = a.dyn_splits ? (int64_t)pl.clusters
                                        : (int64_t)a.splits * a.n_tiles * ((a.m_tiles + pl.cm - 1) / pl.cm);
    const int64_t ncl = std::max<int64_t>(1, std::min<int64_t>(pl.clusters, groups));
    cfg.gridDim = dim3((unsigned)(ncl * pl.cm), 1, 1);
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = dghost::kPdl ? 2 : 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, *static_cast<const CUtensorMap*>(tmA),
                                       *static_cast<const CUtensorMap*>(tmB0), *static_cast<const CUtensorMap*>(tmB1), a);
    dghost::count_launch();
    if (e != cudaSuccess) return DG_ERR_CUDA;
    if (a.splits > 1 || a.dyn_splits) {  // a device plan that does not split leaves the fix-up idle
        const int64_t T = (int64_t)a.m_tiles * a.n_tiles;
        // spread each tile over enough CTAs to give the GPU about 8 per SM, each thread at
        // least one column quad (its partial loads in flight are what hides the latency)
        const int P = dghost::sm_count();
        const bool gu = a.epi == EPI_GELU_GATEUP;
        const int64_t quads = (int64_t)BM * (gu ? C::BN / 2 : C::BN) / 4;
        const unsigned per_tile = (unsigned)std::max<int64_t>(
            1, std::min<int64_t>(std::min<int64_t>(64, quads / 256), (8LL * P + T - 1) / T));
        e = gu ? dghost::launch_pdl(k_fixup<C::BN, true>, dim3((unsigned)T, per_tile, 1), dim3(256), 0, stream, a)
               : dghost::launch_pdl(k_fixup<C::BN, false>, dim3((unsigned)T, per_tile, 1), dim3(256), 0, stream, a);
        dghost::count_launch();
    }
    return dghost::cuda_status(e);
}

// Plan, then launch, with the planned k-slices.
template <class C>
dg_status plan_and_launch(const void* tmA, const void* tmB0, const void* tmB1, GemmArgs a, int64_t max_slots,
                          cudaStream_t stream, int min_slice = 256, int split_below = 101) {
    LaunchPlan pl;
    if (!plan_gemm<C>(a, max_slots, &pl, min_slice, split_below)) return DG_ERR_CUDA;
    a.splits = pl.splits;
    if (a.dyn_splits) {  // the device re-plans for the m-tiles actually active
        a.cm_plan = pl.cm;
        a.clusters = pl.clusters;
        a.min_slice = pl.min_slice;
        a.max_slots = pl.max_slots;
        a.split_below = pl.split_below;
        // j listed canvases: j * tpc active m-tiles (the plan lists whole canvases)
        const int64_t jmax = std::min<int64_t>(kSplitTab, a.tpc > 0 ? a.m_tiles / a.tpc : 0);
        for (int64_t j = 0; j <= jmax; ++j) {
            const int64_t mt = j * a.tpc;
            const int64_t per_split = (int64_t)a.n_tiles * ((mt + pl.cm - 1) / pl.cm);
            a.split_tab[j] = (uint8_t)plan_splits(per_split, mt, a.n_tiles, a.k_blocks, pl.clusters, pl.min_slice,
                                                  pl.max_slots, pl.split_below);
        }
    }
    return launch_gemm<C>(tmA, tmB0, tmB1, a, pl, stream);
}

struct TMaps {
    alignas(64) unsigned char a[128];
    alignas(64) unsigned char b0[128];
    alignas(64) unsigned char b1[128];
};

// 2D bf16 (or fp32) row-major matrix [rows][cols] with row stride ld (elements).
bool tmap_2d(void* tm, int dt, const void* base, int64_t cols, int64_t rows, int64_t ld, uint32_t box_cols,
             uint32_t box_rows, int swz) {
    const int es = dt == 0 ? 2 : 4;
    uint64_t dims[2] = {(uint64_t)cols, (uint64_t)rows};
    uint64_t strides[1] = {(uint64_t)(ld * es)};
    uint32_t box[2] = {box_cols, box_rows};
    return dghost::encode_tmap(tm, dt, 2, const_cast<void*>(base), dims, strides, box, swz);
}

// 3D logits [n][L][ld] as (V, L, n) with box (BK, 128, 1).
bool tmap_logits(void* tm, int dt, const void* base, int64_t V, int32_t L, int64_t n, int64_t ld, uint32_t bk,
                 int swz) {
    const int es = dt == 0 ? 2 : 4;
    uint64_t dims[3] = {(uint64_t)V, (uint64_t)L, (uint64_t)n};
    uint64_t strides[2] = {(uint64_t)(ld * es), (uint64_t)(ld * es * L)};
    uint32_t box[3] = {bk, (uint32_t)BM, 1};
    return dghost::encode_tmap(tm, dt, 3, const_cast<void*>(base), dims, strides, box, swz);
}

struct SelfCondLayout {
    size_t plan, pace, pe, hmid, partial, total;
    int64_t rows;  // compact rows (n * L_pad)
};

SelfCondLayout self_cond_layout(int64_t n, int32_t L, int32_t d, int32_t h, int P) {
    SelfCondLayout l;
    const int tpc = (L + BM - 1) / BM;
    l.rows = n * tpc * BM;
    l.plan = 0;
    l.pace = align256(sizeof(int32_t) * (size_t)(n + 1));
    l.pe = l.pace + 256;
    l.hmid = l.pe + align256((size_t)l.rows * d * 2);
    l.partial = l.hmid + align256((size_t)l.rows * h * 2);
    // partial slots for the P.E GEMM (the only one that splits K)
    const int64_t T = n * tpc * (int64_t)((d + 511) / 512);
    const int64_t slots = T * 32 > 0 ? std::min<int64_t>(T * 32, std::max<int64_t>(T, 8LL * P)) : 0;
    l.total = l.partial + align256((size_t)slots * BM * 512 * 4);
    return l;
}

int64_t pe_partial_slots(int64_t n, int32_t L, int32_t d, int P) {
    const int tpc = (L + BM - 1) / BM;
    const int64_t T = n * tpc * (int64_t)((d + 511) / 512);
    return T * 32 > 0 ? std::min<int64_t>(T * 32, std::max<int64_t>(T, 8LL * P)) : 0;
}

// Smallest k-slice of the self-conditioning GEMMs, in elements of K: a slice of 1024 still
// keeps the tensor cores busy about ten times longer than its partial tile takes to write.
constexpr int kMinSliceK = 1024;

// The three GEMMs of the feedback on compact rows: pe = P.E (already in `pe`), then
// hmid = gelu(pe W_gate^T) * (pe W_up^T), then delta = hmid W_down^T scattered to rows.
// `partial` holds `pe_slots` P.E partial tiles (128 x 512 fp32), i.e. twice as many of the
// MLP's 128 x 256 tiles: a GEMM too small to fill the GPU (under 60 % of its pairs in the
// last round) splits K into them.
dg_status run_mlp(const uint16_t* pe, uint16_t* hmid, int64_t rows, int32_t d, int32_t h, const uint16_t* W_gate,
                  const uint16_t* W_up, const uint16_t* W_down, uint16_t* delta, int64_t delta_ld,
                  const int32_t* plan, int tpc, int32_t L, int32_t m_valid_rows, float* partial, int64_t pe_slots,
                  cudaStream_t stream) {
    const int P = dghost::sm_count();
    TMaps t1, t2;
    if (!tmap_2d(t1.a, 0, pe, d, rows, d, 64, BM, 128)) return DG_ERR_CUDA;
    if (!tmap_2d(t1.b0, 0, W_gate, d, h, d, 64, 128, 128)) return DG_ERR_CUDA;
    if (!tmap_2d(t1.b1, 0, W_up, d, h, d, 64, 128, 128)) return DG_ERR_CUDA;
    GemmArgs g{};
    g.m_tiles = (int32_t)(rows / BM);
    g.plan = plan;
    g.tpc = tpc;
    g.n_tiles = (h + 127) / 128;
    g.k_blocks = (d + 63) / 64;
    g.splits = 1;
    g.K = d;
    g.L = L;
    g.epi = EPI_GELU_GATEUP;
    g.out = hmid;
    g.ldo = h;
    g.n_valid = h;
    g.m_valid = (int32_t)rows;
    g.partial = partial;
    g.status = dghost::status_word();
    const int64_t mlp_slots = partial ? 2 * pe_slots : 0;
    dg_status s = plan_and_launch<GateUp>(t1.a, t1.b0, t1.b1, g, mlp_slots, stream, kMinSliceK / 64, 60);
    if (s != DG_OK) return s;

    if (!tmap_2d(t2.a, 0, hmid, h, rows, h, 64, BM, 128)) return DG_ERR_CUDA;
    if (!tmap_2d(t2.b0, 0, W_down, h, d, h, 64, Down::kPair ? 128 : 256, 128)) return DG_ERR_CUDA;
    GemmArgs q = g;
    q.n_tiles = (d + 255) / 256;
    q.k_blocks = (h + 63) / 64;
    q.K = h;
    q.epi = EPI_SCATTER_BF16;
    q.out = delta;
    q.ldo = delta_ld;
    q.n_valid = d;
    q.m_valid = m_valid_rows;
    (void)P;
    return plan_and_launch<Down>(t2.a, t2.b0, t2.b0, q, mlp_slots, stream, kMinSliceK / 64, 60);
}

dg_status check_weights(int64_t V, int32_t d, int32_t h, const uint16_t* E, const uint16_t* Wg, const uint16_t* Wu,
                        const uint16_t* Wd) {
    if (d < 8 || d > 65536 || h < 8 || h > 65536 || (d % 8) || (h % 8) || V < 2 || V > 0x7fffffffLL)
        return DG_ERR_INVALID_ARG;
    if (!E || !Wg || !Wu || !Wd) return DG_ERR_INVALID_ARG;
    if (!aligned16(E) || !aligned16(Wg) || !aligned16(Wu) || !aligned16(Wd)) return DG_ERR_ALIGNMENT;
    return DG_OK;
}

}  // namespace

// LM head: logits = bf16(hidden . W^T) for the rows of the active canvases, on CTA pairs
// (tcgen05, cta_group::2; 256 x 256 tiles, K = d never split).  With `stats` the epilogue also
// records each row's softmax state per 256-column tile (EPI_LOGIT_STATS).  `plan` holds
// n + 1 ints (the list of active canvases, written here first).
dg_status dghost::lm_head_gemm(const uint16_t* hidden, int64_t ldh, const uint16_t* W, int64_t ldw, int64_t n,
                               int32_t L, int64_t V, int32_t d, const dg_canvas_params* params, uint16_t* logits,
                               int64_t ld, int32_t* plan, float* stats, cudaStream_t stream) {
    cudaError_t e = dghost::launch_pdl(k_plan, dim3(1), dim3(1024), 0, stream, params,
                                       static_cast<const uint8_t*>(nullptr), n, plan, 1);
    dghost::count_launch();
    if (e != cudaSuccess) return DG_ERR_CUDA;
    TMaps tm;
    {
        uint64_t dims[3] = {(uint64_t)d, (uint64_t)L, (uint64_t)n};
        uint64_t strides[2] = {(uint64_t)(ldh * 2), (uint64_t)(ldh * 2 * L)};
        uint32_t box[3] = {64, (uint32_t)BM, 1};
        if (!dghost::encode_tmap(tm.a, 0, 3, const_cast<uint16_t*>(hidden), dims, strides, box, 128))
            return DG_ERR_CUDA;
    }
    if (!tmap_2d(tm.b0, 0, W, d, V, ldw, 64, kLmTileCols / 2, 128)) return DG_ERR_CUDA;
    const int tpc = (L + BM - 1) / BM;
    GemmArgs g{};
    g.m_tiles = (int32_t)(n * tpc);
    g.plan = plan;
    g.tpc = tpc;
    g.n_tiles = (int32_t)((V + kLmTileCols - 1) / kLmTileCols);
    g.k_blocks = (d + 63) / 64;
    g.splits = 1;
    g.K = d;
    g.L = L;
    g.params = params;
    g.epi = stats ? EPI_LOGIT_STATS : EPI_SCATTER_BF16;
    g.out = logits;
    g.ldo = ld;
    g.n_valid = (int32_t)V;
    g.m_valid = (int32_t)(n * tpc * BM);
    g.status = dghost::status_word();
    g.stats = stats;
    g.stats_rows = n * (int64_t)L;
    LaunchPlan pl;
    if (!plan_gemm<LmHead>(g, 0, &pl)) return DG_ERR_CUDA;  // no partial slots: K is never split
    return launch_gemm<LmHead>(tm.a, tm.b0, tm.b0, g, pl, stream);
}

extern "C" {

size_t dg_self_cond_workspace_bytes(int64_t n_canvas, int32_t L, int32_t d, int32_t h) {
    if (n_canvas < 0 || L < 1 || d < 1 || h < 1) return 0;
    const int P = std::max(1, dghost::sm_count());
    return self_cond_layout(n_canvas, L, d, h, P).total;
}

static dg_status self_cond_dims(dg_dtype dtype, int64_t ld, int64_t n_canvas, int32_t L, int64_t V, int32_t d,
                                int32_t h) {
    if (dtype != DG_BF16 && dtype != DG_FP32) return DG_ERR_INVALID_ARG;
    if (n_canvas < 0 || n_canvas > 65535 || L < 1 || L > 1024 || ld < V || V < 2 || V > 0x7fffffffLL)
        return DG_ERR_INVALID_ARG;
    if (d < 8 || d > 65536 || h < 8 || h > 65536 || (d % 8) || (h % 8)) return DG_ERR_INVALID_ARG;
    return DG_OK;
}

// Device-dependent part of the checks (the layout depends on the SM count).
static dg_status self_cond_workspace(int64_t n_canvas, int32_t L, int32_t d, int32_t h, const void* workspace,
                                     size_t workspace_bytes, SelfCondLayout* lay) {
    const int P = dghost::sm_count();
    if (P <= 0) return DG_ERR_CUDA;
    *lay = self_cond_layout(n_canvas, L, d, h, P);
    if (!workspace || workspace_bytes < lay->total) return DG_ERR_WORKSPACE;
    if (!aligned16(workspace)) return DG_ERR_ALIGNMENT;
    return DG_OK;
}

dg_status dg_self_cond_prepare(const dg_canvas_params* params, const uint8_t* converged, int64_t n_canvas,
                               int32_t L, int32_t d, int32_t h, uint16_t* delta_emb, void* workspace,
                               size_t workspace_bytes, dg_stream_t stream) {
    dg_status s = self_cond_dims(DG_BF16, 2, n_canvas, L, 2, d, h);
    if (s != DG_OK || n_canvas == 0) return s;
    if (!params || !delta_emb) return DG_ERR_INVALID_ARG;
    if (!aligned16(delta_emb)) return DG_ERR_ALIGNMENT;
    SelfCondLayout lay;
    s = self_cond_workspace(n_canvas, L, d, h, workspace, workspace_bytes, &lay);
    if (s != DG_OK) return s;
    cudaStream_t st = (cudaStream_t)stream;
    int32_t* plan = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(workspace) + lay.plan);
    // about four CTAs per SM over all canvases (most of them exit at once when feedback is on)
    const int P = std::max(1, dghost::sm_count());
    const int64_t per_canvas = std::max<int64_t>(1, std::min<int64_t>(((int64_t)L * d / 8 + 255) / 256,
                                                                      (4LL * P + n_canvas - 1) / n_canvas));
    dim3 grid((unsigned)per_canvas, (unsigned)n_canvas);
    unsigned* pace = reinterpret_cast<unsigned*>(static_cast<unsigned char*>(workspace) + lay.pace);
    const cudaError_t e = dghost::launch_pdl(k_zero_rows, grid, dim3(256), 0, st, params, converged, n_canvas, L, d,
                                             delta_emb, plan, pace);
    dghost::count_launch();
    return dghost::cuda_status(e);
}

dg_status dg_self_cond_zero_converged(const dg_canvas_params* params, const uint8_t* converged, int64_t n_canvas,
                                      int32_t L, int32_t d, uint16_t* delta_emb, dg_stream_t stream) {
    if (n_canvas < 0 || n_canvas > 65535 || L < 1 || L > 1024 || d < 8 || d > 65536 || (d % 8))
        return DG_ERR_INVALID_ARG;
    if (n_canvas == 0) return DG_OK;
    if (!params || !converged || !delta_emb) return DG_ERR_INVALID_ARG;
    if (!aligned16(delta_emb)) return DG_ERR_ALIGNMENT;
    const int P = std::max(1, dghost::sm_count());
    const int64_t per_canvas = std::max<int64_t>(1, std::min<int64_t>(((int64_t)L * d / 8 + 255) / 256,
                                                                      (4LL * P + n_canvas - 1) / n_canvas));
    const cudaError_t e = dghost::launch_pdl(k_zero_converged, dim3((unsigned)per_canvas, (unsigned)n_canvas),
                                             dim3(256), 0, (cudaStream_t)stream, params, converged, L, d, delta_emb);
    dghost::count_launch();
    return dghost::cuda_status(e);
}

dg_status dg_self_cond_pe(const void* logits, dg_dtype dtype, int64_t ld, const float* lse,
                          const dg_canvas_params* params, int64_t n_canvas, int32_t L, int64_t V, int32_t d,
                          int32_t h, const uint16_t* E, void* workspace, size_t workspace_bytes,
                          dg_stream_t stream) {
    dg_status s = self_cond_dims(dtype, ld, n_canvas, L, V, d, h);
    if (s != DG_OK || n_canvas == 0) return s;
    if (!logits || !lse || !params || !E) return DG_ERR_INVALID_ARG;
    const int es = dtype == DG_BF16 ? 2 : 4;
    if (!aligned16(logits) || (ld * es) % 16 != 0 || !aligned16(E)) return DG_ERR_ALIGNMENT;
    SelfCondLayout lay;
    s = self_cond_workspace(n_canvas, L, d, h, workspace, workspace_bytes, &lay);
    if (s != DG_OK) return s;
    const int P = dghost::sm_count();
    cudaStream_t st = (cudaStream_t)stream;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    const int tpc = (L + BM - 1) / BM;
    // pe = softmax(logits / T) . E  (P formed in shared memory)
    TMaps tm;
    const int bk = 32;
    if (!tmap_logits(tm.a, dtype == DG_BF16 ? 0 : 1, logits, V, L, n_canvas, ld, bk, dtype == DG_BF16 ? 64 : 128))
        return DG_ERR_CUDA;
    if (!tmap_2d(tm.b0, 0, E, d, V, d, 64, bk, 128)) return DG_ERR_CUDA;
    GemmArgs g{};
    g.m_tiles = (int32_t)(n_canvas * tpc);
    g.plan = reinterpret_cast<int32_t*>(ws + lay.plan);
    g.tpc = tpc;
    g.n_tiles = (d + 511) / 512;
    g.k_blocks = (int32_t)((V + bk - 1) / bk);
    g.splits = 1;  // set by the plan
    g.K = V;
    g.L = L;
    g.lse = lse;
    g.params = params;
    g.epi = EPI_BF16;
    g.out = ws + lay.pe;
    g.ldo = d;
    g.n_valid = d;
    g.m_valid = (int32_t)lay.rows;
    g.partial = reinterpret_cast<float*>(ws + lay.partial);
    g.status = dghost::status_word();
    g.dyn_splits = 1;  // the plan lists the canvases with feedback: the device knows how many
    g.pace = reinterpret_cast<unsigned*>(ws + lay.pace);
    const int64_t max_slots = pe_partial_slots(n_canvas, L, d, P);
    return dtype == DG_BF16 ? plan_and_launch<PEbf16>(tm.a, tm.b0, tm.b0, g, max_slots, st, kMinSliceK / bk)
                            : plan_and_launch<PEfp32>(tm.a, tm.b0, tm.b0, g, max_slots, st, kMinSliceK / bk);
}

dg_status dg_self_cond_mlp(int64_t n_canvas, int32_t L, int32_t d, int32_t h, const uint16_t* W_gate,
                           const uint16_t* W_up, const uint16_t* W_down, uint16_t* delta_emb, void* workspace,
                           size_t workspace_bytes, dg_stream_t stream) {
    dg_status s = self_cond_dims(DG_BF16, 2, n_canvas, L, 2, d, h);
    if (s != DG_OK || n_canvas == 0) return s;
    if (!W_gate || !W_up || !W_down || !delta_emb) return DG_ERR_INVALID_ARG;
    if (!aligned16(W_gate) || !aligned16(W_up) || !aligned16(W_down) || !aligned16(delta_emb))
        return DG_ERR_ALIGNMENT;
    SelfCondLayout lay;
    s = self_cond_workspace(n_canvas, L, d, h, workspace, workspace_bytes, &lay);
    if (s != DG_OK) return s;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    const int tpc = (L + BM - 1) / BM;
    const int P = dghost::sm_count();
    return run_mlp(reinterpret_cast<uint16_t*>(ws + lay.pe), reinterpret_cast<uint16_t*>(ws + lay.hmid), lay.rows,
                   d, h, W_gate, W_up, W_down, delta_emb, d, reinterpret_cast<int32_t*>(ws + lay.plan), tpc, L,
                   (int32_t)lay.rows, reinterpret_cast<float*>(ws + lay.partial), pe_partial_slots(n_canvas, L, d, P),
                   (cudaStream_t)stream);
}

dg_status dg_self_cond_logits(const void* logits, dg_dtype dtype, int64_t ld, const float* lse,
                              const dg_canvas_params* params, const uint8_t* converged, int64_t n_canvas, int32_t L,
                              int64_t V, int32_t d, int32_t h, const uint16_t* E, const uint16_t* W_gate,
                              const uint16_t* W_up, const uint16_t* W_down, uint16_t* delta_emb, void* workspace,
                              size_t workspace_bytes, dg_stream_t stream) {
    dg_status s = self_cond_dims(dtype, ld, n_canvas, L, V, d, h);
    if (s != DG_OK) return s;
    s = check_weights(V, d, h, E, W_gate, W_up, W_down);
    if (s != DG_OK) return s;
    if (n_canvas == 0) return DG_OK;
    if (!logits || !lse || !params || !delta_emb) return DG_ERR_INVALID_ARG;
    const int es = dtype == DG_BF16 ? 2 : 4;
    if (!aligned16(logits) || (ld * es) % 16 != 0 || !aligned16(delta_emb)) return DG_ERR_ALIGNMENT;
    SelfCondLayout lay;
    s = self_cond_workspace(n_canvas, L, d, h, workspace, workspace_bytes, &lay);
    if (s != DG_OK) return s;
    s = dg_self_cond_prepare(params, converged, n_canvas, L, d, h, delta_emb, workspace, workspace_bytes, stream);
    if (s != DG_OK) return s;
    s = dg_self_cond_pe(logits, dtype, ld, lse, params, n_canvas, L, V, d, h, E, workspace, workspace_bytes, stream);
    if (s != DG_OK) return s;
    return dg_self_cond_mlp(n_canvas, L, d, h, W_gate, W_up, W_down, delta_emb, workspace, workspace_bytes, stream);
}

size_t dg_self_cond_probs_workspace_bytes(int64_t n_rows, int32_t d, int32_t h) {
    if (n_rows < 0 || d < 1 || h < 1) return 0;
    const int P = std::max(1, dghost::sm_count());
    const int64_t tiles = (n_rows + BM - 1) / BM;
    const int64_t rows = tiles * BM;
    const int64_t T = tiles * ((d + 511) / 512);
    const int64_t slots = T * 32 > 0 ? std::min<int64_t>(T * 32, std::max<int64_t>(T, 8LL * P)) : 0;
    return align256((size_t)rows * d * 2) + align256((size_t)rows * h * 2) + align256((size_t)slots * BM * 512 * 4);
}

dg_status dg_self_cond_probs(const uint16_t* P_rows, int64_t ld, int64_t n_rows, int64_t V, int32_t d, int32_t h,
                             const uint16_t* E, const uint16_t* W_gate, const uint16_t* W_up, const uint16_t* W_down,
                             uint16_t* delta_emb, void* workspace, size_t workspace_bytes, dg_stream_t stream) {
    if (n_rows < 0 || n_rows > (1LL << 24) || ld < V) return DG_ERR_INVALID_ARG;
    dg_status s = check_weights(V, d, h, E, W_gate, W_up, W_down);
    if (s != DG_OK) return s;
    if (n_rows == 0) return DG_OK;
    if (!P_rows || !delta_emb) return DG_ERR_INVALID_ARG;
    if (!aligned16(P_rows) || (ld * 2) % 16 != 0 || !aligned16(delta_emb)) return DG_ERR_ALIGNMENT;
    const size_t need = dg_self_cond_probs_workspace_bytes(n_rows, d, h);
    if (!workspace || workspace_bytes < need) return DG_ERR_WORKSPACE;
    if (!aligned16(workspace)) return DG_ERR_ALIGNMENT;
    const int P = dghost::sm_count();
    if (P <= 0) return DG_ERR_CUDA;
    cudaStream_t st = (cudaStream_t)stream;
    const int64_t tiles = (n_rows + BM - 1) / BM;
    const int64_t rows = tiles * BM;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    uint16_t* pe = reinterpret_cast<uint16_t*>(ws);
    uint16_t* hmid = reinterpret_cast<uint16_t*>(ws + align256((size_t)rows * d * 2));
    float* partial = reinterpret_cast<float*>(ws + align256((size_t)rows * d * 2) + align256((size_t)rows * h * 2));

    TMaps tm;
    const int bk = 32;
    if (!tmap_2d(tm.a, 0, P_rows, V, n_rows, ld, bk, BM, 64)) return DG_ERR_CUDA;
    if (!tmap_2d(tm.b0, 0, E, d, V, d, 64, bk, 128)) return DG_ERR_CUDA;
    GemmArgs g{};
    g.m_tiles = (int32_t)tiles;
    g.plan = nullptr;
    g.tpc = (int32_t)tiles;
    g.n_tiles = (d + 511) / 512;
    g.k_blocks = (int32_t)((V + bk - 1) / bk);
    const int64_t T = (int64_t)g.m_tiles * g.n_tiles;
    const int64_t slots = T * 32 > 0 ? std::min<int64_t>(T * 32, std::max<int64_t>(T, 8LL * P)) : 0;
    g.splits = 1;  // set by the plan
    g.K = V;
    g.L = (int32_t)n_rows;
    g.epi = EPI_BF16;
    g.out = pe;
    g.ldo = d;
    g.n_valid = d;
    g.m_valid = (int32_t)rows;
    g.partial = partial;
    g.status = dghost::status_word();
    s = plan_and_launch<PEprob>(tm.a, tm.b0, tm.b0, g, slots, st);
    if (s != DG_OK) return s;
    return run_mlp(pe, hmid, rows, d, h, W_gate, W_up, W_down, delta_emb, d, nullptr, (int)tiles, (int32_t)n_rows,
                   (int32_t)rows, partial, slots, st);
}

size_t dg_gemm_workspace_bytes(int64_t M, int64_t N) {
    if (M < 1 || N < 1) return 0;
    const int P = std::max(1, dghost::sm_count());
    const int64_t T = ((M + BM - 1) / BM) * ((N + 255) / 256);
    const int64_t slots = std::min<int64_t>(T * 32, std::max<int64_t>(T, 8LL * P));
    return align256((size_t)slots * BM * 512 * 4);
}

dg_status dg_gemm_bf16(const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb, int b_mn_major, float* C,
                       int64_t ldc, int64_t M, int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                       dg_stream_t stream) {
    if (M < 0 || N < 0 || K < 0 || M > (1LL << 24) || N > (1LL << 24) || K > 0x7fffffffLL) return DG_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return DG_OK;
    if (K == 0 || !A || !B || !C || lda < K || ldc < N) return DG_ERR_INVALID_ARG;
    if (b_mn_major ? ldb < N : ldb < K) return DG_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(B) || (lda % 8) || (ldb % 8)) return DG_ERR_ALIGNMENT;
    const size_t need = dg_gemm_workspace_bytes(M, N);
    if (workspace_bytes < need || (need && !workspace)) return DG_ERR_WORKSPACE;
    const int P = dghost::sm_count();
    if (P <= 0) return DG_ERR_CUDA;
    cudaStream_t st = (cudaStream_t)stream;
    TMaps tm;
    GemmArgs g{};
    g.m_tiles = (int32_t)((M + BM - 1) / BM);
    g.tpc = g.m_tiles;
    g.L = (int32_t)M;
    g.epi = EPI_F32;
    g.out = C;
    g.ldo = ldc;
    g.n_valid = (int32_t)N;
    g.m_valid = (int32_t)M;
    g.partial = static_cast<float*>(workspace);
    g.status = dghost::status_word();
    g.K = K;
    const int64_t slots_cap = need / ((size_t)BM * 512 * 4);
    if (b_mn_major) {
        const int bk = 32;
        if (!tmap_2d(tm.a, 0, A, K, M, lda, bk, BM, 64)) return DG_ERR_CUDA;
        if (!tmap_2d(tm.b0, 0, B, N, K, ldb, 64, bk, 128)) return DG_ERR_CUDA;
        g.n_tiles = (int32_t)((N + 511) / 512);
        g.k_blocks = (int32_t)((K + bk - 1) / bk);
        return plan_and_launch<PEprob>(tm.a, tm.b0, tm.b0, g, slots_cap, st);
    }
    const int bk = 64;
    if (!tmap_2d(tm.a, 0, A, K, M, lda, bk, BM, 128)) return DG_ERR_CUDA;
    if (!tmap_2d(tm.b0, 0, B, K, N, ldb, bk, 256, 128)) return DG_ERR_CUDA;
    g.n_tiles = (int32_t)((N + 255) / 256);
    g.k_blocks = (int32_t)((K + bk - 1) / bk);
    return plan_and_launch<DownSingle>(tm.a, tm.b0, tm.b0, g, slots_cap, st);
}

}  // extern "C"

// ------------------------------------------------------------------ no-allocation GEMM
// dg_gemm_bf16_noalloc keeps its split-K partial tiles in this file-scope array instead of a
// caller workspace, for callers that cannot allocate device memory.  Every device that loads
// the library holds the array until the process exits.  Host code must not hand the symbol
// itself to a kernel (on the host it is only a stand-in): the device address is looked up
// once per device with cudaGetSymbolAddress and passed to the kernels.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DG_NOALLOC_SCRATCH_BYTES];

namespace {
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};

// Device address of the scratch array for the current device (looked up on first use).
dg_status noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DG_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return DG_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return DG_OK;
}
}  // namespace

extern "C" dg_status dg_gemm_bf16_noalloc(const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
                                          int b_mn_major, float* C, int64_t ldc, int64_t M, int64_t N, int64_t K,
                                          dg_stream_t stream) {
    if (M < 0 || N < 0 || K < 0 || M > (1LL << 24) || N > (1LL << 24) || K > 0x7fffffffLL) return DG_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return DG_OK;
    if (K == 0 || !A || !B || !C || lda < K || ldc < N) return DG_ERR_INVALID_ARG;
    if (b_mn_major ? ldb < N : ldb < K) return DG_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(B) || (lda % 8) || (ldb % 8)) return DG_ERR_ALIGNMENT;
    const int P = dghost::sm_count();
    if (P <= 0) return DG_ERR_CUDA;
    // the same tiling and k-slices as dg_gemm_bf16, so the two give identical results
    const int bn = b_mn_major ? 512 : 256;
    const int bk = b_mn_major ? 32 : 64;
    GemmArgs g{};
    g.m_tiles = (int32_t)((M + BM - 1) / BM);
    g.tpc = g.m_tiles;
    g.L = (int32_t)M;
    g.epi = EPI_F32;
    g.out = C;
    g.ldo = ldc;
    g.n_valid = (int32_t)N;
    g.m_valid = (int32_t)M;
    g.status = dghost::status_word();
    g.K = K;
    g.n_tiles = (int32_t)((N + bn - 1) / bn);
    g.k_blocks = (int32_t)((K + bk - 1) / bk);
    const int64_t T = (int64_t)g.m_tiles * g.n_tiles;
    const int64_t slots_cap = (int64_t)(dg_gemm_workspace_bytes(M, N) / ((size_t)BM * 512 * 4));
    LaunchPlan pl;
    if (!(b_mn_major ? plan_gemm<PEprob>(g, slots_cap, &pl) : plan_gemm<DownSingle>(g, slots_cap, &pl))) return DG_ERR_CUDA;
    g.splits = pl.splits;
    const size_t need = g.splits > 1 ? (size_t)T * g.splits * BM * bn * 4 : 0;
    if (need > (size_t)DG_NOALLOC_SCRATCH_BYTES) return DG_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    dg_status s = noalloc_scratch(&scratch);
    if (s != DG_OK) return s;
    g.partial = static_cast<float*>(scratch);
    cudaStream_t st = (cudaStream_t)stream;
    TMaps tm;
    if (b_mn_major) {
        if (!tmap_2d(tm.a, 0, A, K, M, lda, bk, BM, 64)) return DG_ERR_CUDA;
        if (!tmap_2d(tm.b0, 0, B, N, K, ldb, 64, bk, 128)) return DG_ERR_CUDA;
        return launch_gemm<PEprob>(tm.a, tm.b0, tm.b0, g, pl, st);
    }
    if (!tmap_2d(tm.a, 0, A, K, M, lda, bk, BM, 128)) return DG_ERR_CUDA;
    if (!tmap_2d(tm.b0, 0, B, K, N, ldb, bk, 256, 128)) return DG_ERR_CUDA;
    return launch_gemm<DownSingle>(tm.a, tm.b0, tm.b0, g, pl, st);
}
