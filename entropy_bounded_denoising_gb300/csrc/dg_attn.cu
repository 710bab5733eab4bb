// dg_attn.cu -- attention with per-sequence causality and a symmetric sliding window, on the
// tensor cores (tcgen05 + TMEM + TMA, sm_103a).
//
// Method (DiffusionGemma vLLM page, sections "시퀀스별로 동적으로 바뀌는 인과 어텐션"
// (per-sequence dynamic causal attention) and "슬라이딩 윈도우 어텐션도 대칭으로" (the sliding
// window made symmetric)): one batch mixes causal requests (prefill and commit passes: query i
// sees keys up to its own position) and bidirectional ones (a denoising canvas: every query
// sees every key of its sequence, context and canvas); attention runs tile by tile and a tile
// holding only masked entries is skipped, saving its MMAs and its K/V reads.  With a window W
// a causal query keeps [pos - W, pos] and a canvas query [pos - W, pos + W].  A sequence's
// queries are its last q_len tokens (query i sits at kv_len - q_len + i); that and the score
// scale * q.k without soft-capping are readings, the pages give only the figures.
//
// Work items are (sequence, 128-query tile, query head); a plan kernel lists the items longest
// first and two persistent CTAs per SM take them, from a counter as they free up when the items
// differ in cost, round robin when they do not (each CTA 256 TMEM columns and under half the
// shared memory, so one CTA's barrier waits are the other's issue slots); one pass with an
// online softmax per item:
//   warp 0      TMA producers: the Q tile once, then K and V tiles (64 keys) in two 2-stage
//               rings (a K buffer frees when its S MMA is done, a V buffer after its P V);
//   warp 1      MMA issuer (one elected thread): S = Q K^T (128 x 64) into TMEM, issued as soon
//               as the softmax has read the previous S, and O += P V with P read from TMEM;
//   warps 2..5  softmax, one query row per thread (its TMEM lane), all 64 columns of a tile:
//               the row of S, the mask on tiles that are not wholly allowed, P = 2^(x - m) as
//               bf16 pairs into one of two TMEM buffers (tcgen05.st) for the P V MMA, the row
//               sum.  The reference m only moves when a row's maximum grows by more than 8 (in
//               log2 units), so P < 2^8 and most tiles leave O alone; when it moves, the row of
//               O is rescaled in TMEM (tcgen05.ld, multiply, tcgen05.st) after the last P V.
//               At the end O / l goes out in bf16 with the row's lse.
// Only key tiles holding an allowed key for some query of the tile are visited.
#include <cuda.h>
#include <cuda_runtime.h>

#include <math.h>

#include <algorithm>

#include "dg_common.cuh"

namespace {

constexpr int kTile = 128;      // queries per CTA
constexpr int kKeys = 64;       // keys per tile
constexpr int kSub = 64;        // columns per 128-byte swizzle atom
constexpr uint32_t kQSub = kTile * kSub * 2;       // 16 KB: 128 rows x 64 columns of Q
constexpr uint32_t kKSub = kKeys * kSub * 2;       // 8 KB: 64 rows x 64 columns of K or V
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
#ifndef DG_ATTN_RESCALE_LOG2
#define DG_ATTN_RESCALE_LOG2 8
#endif
constexpr float kRescaleAbove = DG_ATTN_RESCALE_LOG2;  // log2 units: P < 2^this between rescales

struct AttnArgs {
    const int32_t* cu_q;    // [n + 1] query offsets
    const int32_t* cu_kv;   // [n + 1] key offsets
    const uint8_t* causal;  // [n]
    uint16_t* o;            // [total_q][Hq][D] bf16
    float* lse;             // [total_q][Hq] or null
    int32_t Hq, Hkv, window;
    int64_t total_q, total_kv;
    float scale_log2;       // scale * log2(e)
    unsigned* status;
};

struct __align__(8) AttnShared {
    uint64_t qfull;
    uint64_t qempty;          // the Q tile has been read by the item's last S MMA
    uint64_t oempty;          // the softmax has read O out for the item (the next may overwrite it)
    uint64_t kfull[2];        // K and V tiles in separate rings: a K buffer is free as soon as
    uint64_t kempty[2];       // its S MMA is done, long before the V buffer of the same tile
    uint64_t vfull[2];
    uint64_t vempty[2];
    uint64_t sfull;
    uint64_t sempty;
    uint64_t pfull[2];        // P buffer b written by the four softmax warps (one barrier per buffer:
                              // with one for both, a warp a tile ahead could complete the phase of
                              // a tile whose P another warp is still writing)
    uint64_t pvdone[2];       // P V of the tiles using P buffer 0 / 1 done
    uint64_t mmadone;
    uint64_t wfull[4];        // the item queue: slot k % 4 holds the CTA's k-th work index
    uint64_t wempty[4];       // (-1: no more), taken by its 7 readers
    int64_t item_w[4];
    uint32_t tmem_base;
    int abort_flag;
};

// Per head dimension D (64, 128 or 256): shared memory Q | K[2] | V[2] (1024-aligned blocks of
// D / 64 swizzle atoms each), then the barriers; tensor memory columns S (64), O (D), the two P
// buffers (bf16 pairs: 32 columns for 64 keys each), rounded up to a power of two.  Two CTAs
// share an SM while both fit (D = 64, 128), else one (D = 256).
template <int D>
struct AttnCfg {
    static_assert(D == 64 || D == 128 || D == 256, "head dimension 64, 128 or 256");
    static constexpr int kHead = D;
    static constexpr uint32_t kQBytes = (D / kSub) * kQSub;     // the Q tile
    static constexpr uint32_t kKVBytes = (D / kSub) * kKSub;    // one K (or V) tile
    static constexpr uint32_t kOffQ = 0;
    static constexpr uint32_t kOffK = kOffQ + kQBytes;
    static constexpr uint32_t kOffV = kOffK + 2 * kKVBytes;
    static constexpr uint32_t kOffBar = kOffV + 2 * kKVBytes;
    static constexpr size_t kSmem = 1024 + kOffBar + sizeof(AttnShared) + 64;
    static constexpr uint32_t kColS = 0, kColO = 64, kColP = 64 + D;
    static constexpr uint32_t kTmemCols = (kColP + 64 <= 256) ? 256 : 512;
    static constexpr int kCtasPerSm = (2 * (kSmem + 1024) <= 232448 && 2 * kTmemCols <= 512) ? 2 : 1;
    static_assert(kSmem <= 232448, "fits the opt-in shared memory of an SM");
};
constexpr int kThreads = 192;

// The key tiles a query tile visits, and whether a key tile is allowed for all its queries.
struct TileRange {
    int q0, ql, k0, kl;   // sequence offsets and lengths
    int pmin, pmax;       // positions of the tile's first and last real query
    int jt_lo, nt;        // first key tile and count
    bool causal;
};

DG_DEVINL TileRange tile_range(const AttnArgs& a, int s, int t) {
    TileRange r;
    r.q0 = a.cu_q[s];
    r.ql = a.cu_q[s + 1] - r.q0;
    r.k0 = a.cu_kv[s];
    r.kl = a.cu_kv[s + 1] - r.k0;
    r.causal = a.causal[s] != 0;
    const int off = r.kl - r.ql;
    r.pmin = off + t * kTile;
    r.pmax = off + min(r.ql, t * kTile + kTile) - 1;
    const int64_t W = a.window;
    const int jlo = W >= 0 ? (int)max((int64_t)0, (int64_t)r.pmin - W) : 0;
    const int jhi = r.causal ? r.pmax : (W >= 0 ? (int)min((int64_t)r.kl - 1, (int64_t)r.pmax + W) : r.kl - 1);
    r.jt_lo = jlo / kKeys;
    r.nt = jhi >= jlo ? jhi / kKeys - r.jt_lo + 1 : 0;
    return r;
}

DG_DEVINL bool tile_full(const TileRange& r, int window, int jt) {
    const int64_t j0 = (int64_t)jt * kKeys, j1 = j0 + kKeys - 1;
    if (j1 >= r.kl) return false;
    if (r.causal && j1 > r.pmin) return false;
    if (window >= 0) {
        if (j0 < (int64_t)r.pmax - window) return false;
        if (!r.causal && j1 > (int64_t)r.pmin + window) return false;
    }
    return true;
}

DG_DEVINL uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t v;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(v) : "f"(hi), "f"(lo));
    return v;
}

DG_DEVINL float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed fp32 pairs (one rounding per element, as the scalar forms).
DG_DEVINL uint64_t f2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
DG_DEVINL void f2_split(uint64_t v, float& a, float& b) { asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v)); }
DG_DEVINL uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
DG_DEVINL uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// Barrier waits on the per-tile critical path: a 200 ns suspend-time hint (measured against
// none, which lets a polling lane take issue slots from the other softmax warp, and 1000 ns,
// which wakes late next to this loop's ~2 us per tile); bounded.
#ifndef DG_ATTN_HINT_NS
#define DG_ATTN_HINT_NS 200
#endif
DG_DEVINL bool attn_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
#if DG_ATTN_HINT_NS > 0
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(dg::smem_u32(bar)), "r"(parity), "r"((uint32_t)DG_ATTN_HINT_NS)
        : "memory");
#else
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(dg::smem_u32(bar)), "r"(parity)
        : "memory");
#endif
    return ok != 0;
}

DG_DEVINL bool attn_wait(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < 4u * dg::kWaitPolls; ++i)
        if (attn_try_wait(bar, parity)) return true;
    return false;
}

// Whole warp: lane 0 polls, then the warp synchronises.
DG_DEVINL bool attn_wait_warp(uint64_t* bar, uint32_t parity) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = attn_wait(bar, parity) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();
    return ok != 0;
}

DG_DEVINL bool aborted(const AttnShared& sh) { return *(volatile const int*)&sh.abort_flag != 0; }

// Which items a CTA works.  When they all cost the same, CTA b takes b, b + grid, ...: with two
// CTAs per SM that spreads the last round over distinct SMs (claiming from a counter lets both
// CTAs of an SM, which finish together, take the last items together).  When they differ, the
// CTA's Q producer claims the next work index from a launch-wide counter once the Q buffer
// frees (later claims balance better: a CTA holds at most the item it is computing and the
// claimed one, and CTAs that finish early take more; the items are ordered longest first) and
// publishes it in the CTA's item queue, where the K and V producers, the MMA issuer and the
// four softmax warps read it in turn.
constexpr int kQueueReaders = 7;

DG_DEVINL int64_t take_item(AttnShared& sh, uint32_t k, bool& ok) {
    const int slot = (int)(k & 3u);
    if (!attn_wait(&sh.wfull[slot], (k >> 2) & 1u)) {
        ok = false;
        return -1;
    }
    const int64_t w = *(volatile int64_t*)&sh.item_w[slot];
    dg::mbar_arrive(&sh.wempty[slot]);
    return w;
}

DG_DEVINL int64_t take_item_warp(AttnShared& sh, uint32_t k, bool& ok) {
    const int slot = (int)(k & 3u);
    if (!attn_wait_warp(&sh.wfull[slot], (k >> 2) & 1u)) {
        ok = false;
        return -1;
    }
    const int64_t w = *(volatile int64_t*)&sh.item_w[slot];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) dg::mbar_arrive(&sh.wempty[slot]);
    return w;
}

DG_DEVINL void do_abort(AttnShared& sh, unsigned* status) {
    *(volatile int*)&sh.abort_flag = 1;
    dg::raise_status(status, DG_DEV_TIMEOUT);
}

// ------------------------------------------------------------------ the plan
// Work items are (sequence, 128-query tile) pairs with at least one query.  One CTA lists them
// by decreasing cost (key tiles visited; a counting sort over kCostBuckets), so that the
// persistent CTAs, which take items in that order, start with the longest.  A sequence whose
// offsets or lengths are out of range, or that has more queries than max_q_tiles tiles hold,
// raises DG_DEV_BAD_PARAM and is left out (wholly, or its tiles past max_q_tiles).
constexpr int kCostBuckets = 1024;
constexpr int kPlanHeader = 4;  // ints before the items: the item count, a one-cost flag, a 64-bit work counter

__global__ void __launch_bounds__(1024) k_attn_plan(const AttnArgs a, int32_t n_seq, int32_t max_q_tiles,
                                                    int32_t* __restrict__ plan) {
    __shared__ int count[kCostBuckets];
    __shared__ int warp_sum[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int b = tid; b < kCostBuckets; b += blockDim.x) count[b] = 0;
    if (tid == 0) *reinterpret_cast<unsigned long long*>(plan + 2) = 0ull;  // the attention kernel's work counter
    __syncthreads();
    const int64_t pairs = (int64_t)n_seq * max_q_tiles;
    auto item_key = [&](int64_t f, int& key) -> bool {  // false: no item (past the queries or bad)
        const int s = (int)(f / max_q_tiles), t = (int)(f % max_q_tiles);
        const TileRange r = tile_range(a, s, t);
        const bool bad = r.q0 < 0 || r.k0 < 0 || r.ql < 0 || (int64_t)r.q0 + r.ql > a.total_q ||
                         (int64_t)r.k0 + r.kl > a.total_kv || r.ql > r.kl;
        if (t == 0 && (bad || r.ql > max_q_tiles * kTile)) dg::raise_status(a.status, DG_DEV_BAD_PARAM);
        if (bad || t * kTile >= r.ql || r.nt <= 0) return false;
        key = kCostBuckets - 1 - min(r.nt, kCostBuckets - 1);  // longest first
        return true;
    };
    for (int64_t f = tid; f < pairs; f += blockDim.x) {
        int key;
        if (item_key(f, key)) atomicAdd(&count[key], 1);
    }
    __syncthreads();
    // exclusive prefix over the buckets (one per thread): warp scans, then the warp totals
    const int c = tid < kCostBuckets ? count[tid] : 0;
    // items of one cost: the kernel's CTAs take them round robin (balanced per SM), else from
    // the counter (list scheduling, longest first)
    const int n_costs = __syncthreads_count(c > 0);
    if (tid == 0) plan[1] = n_costs <= 1 ? 1 : 0;
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int v = warp_sum[lane];
        int wi = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += y;
        }
        warp_sum[lane] = wi - v;
        if (lane == 31) plan[0] = wi;
    }
    __syncthreads();
    if (tid < kCostBuckets) count[tid] = warp_sum[warp] + incl - c;
    __syncthreads();
    int2* items = reinterpret_cast<int2*>(plan + kPlanHeader);
    for (int64_t f = tid; f < pairs; f += blockDim.x) {
        int key;
        if (item_key(f, key)) items[atomicAdd(&count[key], 1)] = make_int2((int)(f / max_q_tiles), (int)(f % max_q_tiles));
    }
}

// ------------------------------------------------------------------ the kernel
// Persistent: the CTAs take work indices w of n_items * Hq (item w / Hq, head w % Hq) in the
// plan's order (longest first), round robin or from the counter through the item queue (see
// above).  Every ring, buffer and barrier phase is counted over the CTA's whole run (g: its key
// tiles so far, k: its items so far), so the next item's Q and K / V loads and its first S MMA
// overlap the current item's last tiles and its epilogue.
template <int D>
__global__ void __launch_bounds__(kThreads, AttnCfg<D>::kCtasPerSm)
    k_attention(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const AttnArgs a, const int32_t* __restrict__ plan) {
    using C = AttnCfg<D>;
    constexpr int kHead = D;
    constexpr uint32_t kQBytes = C::kQBytes, kKVBytes = C::kKVBytes;
    constexpr uint32_t kOffQ = C::kOffQ, kOffK = C::kOffK, kOffV = C::kOffV, kOffBar = C::kOffBar;
    constexpr uint32_t kColS = C::kColS, kColO = C::kColO, kColP = C::kColP, kTmemCols = C::kTmemCols;
    extern __shared__ __align__(1024) unsigned char attn_smem_raw[];
    unsigned char* smem =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(attn_smem_raw) + 1023) & ~uintptr_t(1023));
    AttnShared& sh = *reinterpret_cast<AttnShared*>(smem + kOffBar);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n_work = (int64_t)plan[0] * a.Hq;
    if ((int64_t)blockIdx.x >= n_work) return;  // the whole CTA: no work
    const int2* items = reinterpret_cast<const int2*>(plan + kPlanHeader);
    const int group = a.Hq / a.Hkv;
    const bool round_robin = plan[1] != 0;
    auto rr_item = [&](uint32_t k) -> int64_t {
        const int64_t w = (int64_t)blockIdx.x + (int64_t)k * gridDim.x;
        return w < n_work ? w : -1;
    };

    if (threadIdx.x == 0) {
        dg::mbar_init(&sh.qfull, 1);
        dg::mbar_init(&sh.qempty, 1);
        dg::mbar_init(&sh.oempty, 4);  // one arrival per softmax warp
        for (int i = 0; i < 2; ++i) {
            dg::mbar_init(&sh.kfull[i], 1);
            dg::mbar_init(&sh.kempty[i], 1);
            dg::mbar_init(&sh.vfull[i], 1);
            dg::mbar_init(&sh.vempty[i], 1);
            dg::mbar_init(&sh.pvdone[i], 1);
        }
        dg::mbar_init(&sh.sfull, 1);
        dg::mbar_init(&sh.sempty, 4);
        dg::mbar_init(&sh.pfull[0], 4);
        dg::mbar_init(&sh.pfull[1], 4);
        dg::mbar_init(&sh.mmadone, 1);
        for (int i = 0; i < 4; ++i) {
            dg::mbar_init(&sh.wfull[i], 1);
            dg::mbar_init(&sh.wempty[i], kQueueReaders);
        }
        sh.abort_flag = 0;
        dg::fence_mbar_init();
    }
    if (warp == 1) {
        dg::tmem_alloc(&sh.tmem_base, kTmemCols);
        dg::tmem_relinquish();
    }
    dg::tc_fence_before();
    __syncthreads();
    dg::tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    const uint32_t sQ = dg::smem_u32(smem + kOffQ);

    if (warp == 0) {
        // ------------------------------------------------ TMA producers: lane 0 the K ring, lane 1
        // the V ring, lane 2 the Q tile of each item (once the last item's last S has read it)
        if (lane == 2) {
            dg::prefetch_tmap(&tmQ);
            unsigned long long* counter = reinterpret_cast<unsigned long long*>(const_cast<int32_t*>(plan) + 2);
            uint32_t kq = 0;
            bool ok = true;
            for (;; ++kq) {
                const int slot = (int)(kq & 3u);
                if (!attn_wait(&sh.qempty, (kq & 1u) ^ 1u) ||
                    (!round_robin && !attn_wait(&sh.wempty[slot], ((kq >> 2) & 1u) ^ 1u))) {
                    ok = false;
                    break;
                }
                int64_t w;
                if (round_robin) {
                    w = rr_item(kq);
                } else {
                    w = (int64_t)atomicAdd(counter, 1ull);
                    if (w >= n_work || aborted(sh)) w = -1;
                    sh.item_w[slot] = w;
                    dg::mbar_arrive(&sh.wfull[slot]);  // releases the index to the readers
                }
                if (w < 0 || aborted(sh)) break;
                const int2 it = items[w / a.Hq];
                const int h = (int)(w % a.Hq);
                const int qrow = a.cu_q[it.x] + it.y * kTile;
                dg::mbar_arrive_expect_tx(&sh.qfull, kQBytes);
#pragma unroll
                for (int c = 0; c < kHead / kSub; ++c)
                    dg::tma_load_2d(smem + kOffQ + c * kQSub, &tmQ, h * kHead + c * kSub, qrow, &sh.qfull);
            }
            if (!ok) do_abort(sh, a.status);
            if (aborted(sh) && kq > 0) (void)attn_wait(&sh.qfull, (kq - 1u) & 1u);  // the last Q copy landed
        } else if (lane < 2) {
            const bool is_k = lane == 0;
            const CUtensorMap* tm = is_k ? &tmK : &tmV;
            uint64_t* full = is_k ? sh.kfull : sh.vfull;
            uint64_t* empty = is_k ? sh.kempty : sh.vempty;
            unsigned char* ring = smem + (is_k ? kOffK : kOffV);
            dg::prefetch_tmap(tm);
            uint32_t g = 0;
            int issued[2] = {0, 0};
            bool ok = true;
            for (uint32_t k = 0; ok && !aborted(sh); ++k) {
                const int64_t w = round_robin ? rr_item(k) : take_item(sh, k, ok);
                if (w < 0) break;
                const int2 it = items[w / a.Hq];
                const int hk = (int)(w % a.Hq) / group;
                const TileRange r = tile_range(a, it.x, it.y);
                for (int i = 0; i < r.nt; ++i, ++g) {
                    const int st = (int)(g & 1u);
                    if (!attn_wait(&empty[st], ((g >> 1) & 1u) ^ 1u)) {
                        ok = false;
                        break;
                    }
                    dg::mbar_arrive_expect_tx(&full[st], kKVBytes);
                    const int krow = r.k0 + (r.jt_lo + i) * kKeys;
                    unsigned char* dst = ring + st * kKVBytes;
#pragma unroll
                    for (int c = 0; c < kHead / kSub; ++c)
                        dg::tma_load_2d(dst + c * kKSub, tm, hk * kHead + c * kSub, krow, &full[st]);
                    ++issued[st];
                }
            }
            if (!ok) do_abort(sh, a.status);
            if (aborted(sh)) {  // never leave with a copy still landing in shared memory
                for (int st = 0; st < 2; ++st)
                    if (issued[st] > 0) (void)attn_wait(&full[st], (uint32_t)(issued[st] - 1) & 1u);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = dg::instr_desc(kTile, kKeys, false);  // S = Q K^T: K tile K-major
            constexpr uint32_t idO = dg::instr_desc(kTile, kHead, true);   // O += P V: V rows are N-major
            uint32_t g = 0, kq = 0;
            bool ok = true;
            for (; ok && !aborted(sh); ++kq) {
                const int64_t w = round_robin ? rr_item(kq) : take_item(sh, kq, ok);
                if (w < 0) break;
                const int2 it = items[w / a.Hq];
                const TileRange r = tile_range(a, it.x, it.y);
                if (!attn_wait(&sh.qfull, kq & 1u)) {
                    ok = false;
                    break;
                }
                for (int i = 0; i <= r.nt; ++i) {
                    if (i < r.nt) {  // S of tile g + i, once the softmax has read the previous S
                        const uint32_t gs = g + (uint32_t)i;
                        const int st = (int)(gs & 1u);
                        if (!attn_wait(&sh.kfull[st], (gs >> 1) & 1u) || !attn_wait(&sh.sempty, (gs & 1u) ^ 1u)) {
                            ok = false;
                            break;
                        }
                        dg::tc_fence_after();
                        const uint32_t sK = dg::smem_u32(smem + kOffK + st * kKVBytes);
#pragma unroll
                        for (int kk = 0; kk < kHead / 16; ++kk) {
                            const uint32_t offq = (uint32_t)(kk >> 2) * kQSub + (uint32_t)(kk & 3) * 32u;
                            const uint32_t offk = (uint32_t)(kk >> 2) * kKSub + (uint32_t)(kk & 3) * 32u;
                            dg::tc_mma_f16(tmem + kColS, dg::smem_desc(sQ + offq, 16, 1024, 128),
                                           dg::smem_desc(sK + offk, 16, 1024, 128), idS, kk > 0 ? 1u : 0u);
                        }
                        dg::tc_commit(&sh.sfull);
                        dg::tc_commit(&sh.kempty[st]);              // the K buffer, once S has read it
                        if (i == r.nt - 1) dg::tc_commit(&sh.qempty);  // the Q buffer, after the item's last S
                    }
                    if (i >= 1) {  // O += P V of tile g + i - 1 once the softmax has written P
                        const int j = i - 1;
                        const uint32_t gp = g + (uint32_t)j;
                        const int st = (int)(gp & 1u);
                        if (!attn_wait(&sh.pfull[st], (gp >> 1) & 1u) || !attn_wait(&sh.vfull[st], (gp >> 1) & 1u) ||
                            (j == 0 && !attn_wait(&sh.oempty, (kq & 1u) ^ 1u))) {  // the last item's O read out
                            ok = false;
                            break;
                        }
                        dg::tc_fence_after();
                        const uint32_t sV = dg::smem_u32(smem + kOffV + st * kKVBytes);
#pragma unroll
                        for (int kk = 0; kk < kKeys / 16; ++kk) {
                            // A: P in tensor memory, 16 keys = 8 columns per step; B: 16 V rows (keys)
                            // x D columns (D / 64 atoms of 64 columns, kKSub apart)
                            dg::tc_mma_f16_ts(tmem + kColO, tmem + kColP + (uint32_t)(st * 32 + kk * 8),
                                              dg::smem_desc(sV + (uint32_t)kk * 16u * 128u, kKSub, 1024, 128), idO,
                                              (j > 0 || kk > 0) ? 1u : 0u);
                        }
                        dg::tc_commit(&sh.pvdone[st]);
                        dg::tc_commit(&sh.vempty[st]);
                    }
                }
                g += (uint32_t)r.nt;
            }
            if (!ok) do_abort(sh, a.status);
            // every MMA issued above has completed before the tensor memory is released
            dg::tc_commit(&sh.mmadone);
            (void)attn_wait(&sh.mmadone, 0);
        }
    } else {
        // ------------------------------------------------ softmax (warps 2..5), one row per thread
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        const int row = q * 32 + lane;
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        uint32_t g = 0, kq = 0;
        bool ok = true;
        for (; ok; ++kq) {
            const int64_t w = round_robin ? rr_item(kq) : take_item_warp(sh, kq, ok);
            if (w < 0) break;
            const int2 it = items[w / a.Hq];
            const int h = (int)(w % a.Hq);
            const TileRange r = tile_range(a, it.x, it.y);
            const int t = it.y;
            const int pos = r.kl - r.ql + t * kTile + row;
            const bool row_valid = t * kTile + row < r.ql;
            float m_ref = -INFINITY, l = 0.f;
            for (int i = 0; i < r.nt; ++i) {
                const uint32_t gi = g + (uint32_t)i;
                if (!attn_wait_warp(&sh.sfull, gi & 1u)) {
                    ok = false;
                    break;
                }
                dg::tc_fence_after();
                float x[2][32];
                {
                    uint32_t raw[2][32];
#pragma unroll
                    for (int c = 0; c < 2; ++c) dg::tmem_ld32_nowait(tmem + lane_base + kColS + (uint32_t)(c * 32), raw[c]);
                    dg::tmem_ld_wait_dep(raw[0]);
                    dg::tmem_ld_wait_dep(raw[1]);  // (returns at once: no load is left in flight)
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int e = 0; e < 32; ++e) x[c][e] = __uint_as_float(raw[c][e]);
                }
                dg::tc_fence_before();
                __syncwarp();
                if (lane == 0) dg::mbar_arrive(&sh.sempty);  // S free for the next tile's S
                const int jt = r.jt_lo + i;
                const int j0 = jt * kKeys;
                if (!tile_full(r, a.window, jt)) {
                    // masked entries: -inf, which 2^x maps to 0.  The keys a query at position pos may
                    // see form one range: j < kv_len, j <= pos if causal, and with a window W also
                    // j >= pos - W and (bidirectional) j <= pos + W; the mask is two compares per entry
                    const int64_t W = a.window;
                    const int lo = (int)max((int64_t)-1, (W >= 0 ? (int64_t)pos - W : 0) - j0);
                    const int hi = (int)min((int64_t)kKeys,
                                            min((int64_t)r.kl - 1, r.causal ? (int64_t)pos : (W >= 0 ? (int64_t)pos + W : (int64_t)r.kl - 1)) - j0);
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int kx = c * 32 + e;
                            x[c][e] = (kx >= lo && kx <= hi) ? x[c][e] : -INFINITY;
                        }
                }
                // the tile's row maximum of the raw scores (a tree: independent steps), in log2 units
                float mx[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) mx[e] = fmaxf(fmaxf(x[0][2 * e], x[0][2 * e + 1]), fmaxf(x[1][2 * e], x[1][2 * e + 1]));
#pragma unroll
                for (int wd = 8; wd >= 1; wd >>= 1)
#pragma unroll
                    for (int e = 0; e < wd; ++e) mx[e] = fmaxf(mx[e], mx[e + wd]);
                const float tmax = mx[0] * a.scale_log2;  // -inf stays -inf (scale > 0)
                const bool rescale = __any_sync(0xffffffffu, tmax > m_ref + kRescaleAbove);  // m_ref = -inf: any finite max
                // O is rescaled only after this item's last P V (which implies the one before);
                // otherwise P buffer gi % 2 must have been read by the P V two tiles back, which may
                // be the previous item's
                if ((rescale && i > 0) || gi > 1) {
                    const uint32_t gj = (rescale && i > 0) ? gi - 1 : gi - 2;
                    if (!attn_wait_warp(&sh.pvdone[gj & 1u], (gj >> 1) & 1u)) {
                        ok = false;
                        break;
                    }
                    dg::tc_fence_after();
                }
                if (rescale) {
                    const float m_new = fmaxf(m_ref, tmax);
                    const float alpha = (m_new == -INFINITY) ? 1.f : ex2(m_ref - m_new);
                    l *= alpha;
                    if (i > 0) {
#pragma unroll
                        for (int c = 0; c < kHead / 32; ++c) {
                            float o[32];
                            const uint32_t ta = tmem + lane_base + kColO + (uint32_t)(c * 32);
                            dg::tmem_ld32(ta, o);
#pragma unroll
                            for (int e = 0; e < 32; ++e) o[e] *= alpha;
                            dg::tmem_st32(ta, o);
                            dg::tmem_st_wait();  // before the next chunk's load may reuse the registers
                        }
                    }
                    m_ref = m_new;
                }
                // P = 2^(s c - m_ref) in bf16 pairs into P buffer gi % 2 for the P V MMA; the exponent
                // in one packed fma per pair (a row with no allowed key yet keeps m_ref = -inf: its
                // entries are all -inf and the offset 0 keeps them so)
                const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;
                const uint64_t cc = f2(a.scale_log2, a.scale_log2), mm = f2(neg_m, neg_m);
                uint64_t acc = f2(0.f, 0.f);
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        float z0, z1;
                        f2_split(f2_fma(f2(x[c][e], x[c][e + 1]), cc, mm), z0, z1);
                        const float p0 = ex2(z0), p1 = ex2(z1);
                        acc = f2_add(acc, f2(p0, p1));
                        pk[c * 16 + e / 2] = pack_bf16x2(p0, p1);
                    }
                }
                float sa, sb;
                f2_split(acc, sa, sb);
                dg::tmem_st32u(tmem + lane_base + kColP + (gi & 1u) * 32u, pk);
                dg::tmem_st_wait();
                l += sa + sb;
                dg::tc_fence_before();
                __syncwarp();
                if (lane == 0) dg::mbar_arrive(&sh.pfull[gi & 1u]);
            }
            if (!ok) break;
            const uint32_t gl = g + (uint32_t)r.nt - 1u;  // the item's last P V
            if (!attn_wait_warp(&sh.pvdone[gl & 1u], (gl >> 1) & 1u)) {
                ok = false;
                break;
            }
            dg::tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const int64_t qi = (int64_t)r.q0 + t * kTile + row;
            uint16_t* orow = a.o + (qi * a.Hq + h) * kHead;
#pragma unroll
            for (int c = 0; c < kHead / 32; ++c) {
                float o[32];
                dg::tmem_ld32(tmem + lane_base + kColO + (uint32_t)(c * 32), o);
                if (row_valid) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8)
                        *reinterpret_cast<uint4*>(orow + c * 32 + e) =
                            make_uint4(pack_bf16x2(o[e] * inv, o[e + 1] * inv), pack_bf16x2(o[e + 2] * inv, o[e + 3] * inv),
                                       pack_bf16x2(o[e + 4] * inv, o[e + 5] * inv), pack_bf16x2(o[e + 6] * inv, o[e + 7] * inv));
                }
            }
            if (row_valid && a.lse) a.lse[qi * a.Hq + h] = (m_ref + log2f(l)) * kLn2;
            dg::tc_fence_before();
            __syncwarp();
            if (lane == 0) dg::mbar_arrive(&sh.oempty);  // O read out: the next item may overwrite it
            g += (uint32_t)r.nt;
        }
        if (!ok) do_abort(sh, a.status);
    }

    dg::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        dg::tc_fence_after();
        dg::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

// ------------------------------------------------------------------ host side
namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// [rows][heads * D] bf16 with boxes of 64 columns (one 128-byte swizzle atom) x box_rows.
bool tmap_heads(CUtensorMap* tm, const void* base, int64_t rows, int32_t heads, int32_t D, uint32_t box_rows) {
    uint64_t dims[2] = {(uint64_t)heads * D, (uint64_t)rows};
    uint64_t strides[1] = {(uint64_t)heads * D * 2};
    uint32_t box[2] = {(uint32_t)kSub, box_rows};
    return dghost::encode_tmap(tm, 0, 2, const_cast<void*>(base), dims, strides, box, 128);
}

// Plan: a header and one (sequence, query tile) entry per possible item.
size_t plan_bytes(int64_t n_seq, int64_t max_q_tiles) {
    return ((size_t)kPlanHeader * 4 + (size_t)n_seq * (size_t)max_q_tiles * 8 + 255) / 256 * 256;
}

}  // namespace

extern "C" size_t dg_attention_workspace_bytes(int32_t n_seq, int32_t max_q_len) {
    if (n_seq < 0 || max_q_len < 1) return 0;
    return plan_bytes(n_seq, (max_q_len + kTile - 1) / kTile);
}

extern "C" dg_status dg_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o, float* lse,
                                  const int32_t* cu_q, const int32_t* cu_kv, const uint8_t* causal, int32_t n_seq,
                                  int32_t max_q_len, int64_t total_q, int64_t total_kv, int32_t Hq, int32_t Hkv,
                                  int32_t D, int32_t window, float scale, void* workspace, size_t workspace_bytes,
                                  dg_stream_t stream) {
    if (n_seq < 0 || n_seq > 65535 || Hq < 1 || Hq > 65535 || Hkv < 1 || Hq % Hkv != 0 || window < -1 ||
        !(scale == scale) || scale == INFINITY || scale == -INFINITY)
        return DG_ERR_INVALID_ARG;
    if (D != 64 && D != 128 && D != 256) return DG_ERR_UNSUPPORTED;
    if (n_seq == 0) return DG_OK;
    if (max_q_len < 1 || max_q_len > (1 << 30) || total_q < 1 || total_kv < 1 || total_q >= (1LL << 31) ||
        total_kv >= (1LL << 31))
        return DG_ERR_INVALID_ARG;
    if (!q || !k || !v || !o || !cu_q || !cu_kv || !causal) return DG_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return DG_ERR_ALIGNMENT;
    const int32_t max_q_tiles = (max_q_len + kTile - 1) / kTile;
    if (!workspace || workspace_bytes < plan_bytes(n_seq, max_q_tiles)) return DG_ERR_WORKSPACE;
    if (!aligned16(workspace)) return DG_ERR_ALIGNMENT;
    const int P = dghost::sm_count();
    if (P <= 0) return DG_ERR_CUDA;
    CUtensorMap tq, tk, tv;
    if (!tmap_heads(&tq, q, total_q, Hq, D, kTile) || !tmap_heads(&tk, k, total_kv, Hkv, D, kKeys) ||
        !tmap_heads(&tv, v, total_kv, Hkv, D, kKeys))
        return DG_ERR_CUDA;
    AttnArgs a;
    a.cu_q = cu_q;
    a.cu_kv = cu_kv;
    a.causal = causal;
    a.o = o;
    a.lse = lse;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.window = window;
    a.total_q = total_q;
    a.total_kv = total_kv;
    a.scale_log2 = scale * kLog2e;
    a.status = dghost::status_word();
    int32_t* plan = static_cast<int32_t*>(workspace);
    cudaStream_t st = (cudaStream_t)stream;
    k_attn_plan<<<1, 1024, 0, st>>>(a, n_seq, max_q_tiles, plan);
    dghost::count_launch();
    if (cudaGetLastError() != cudaSuccess) return DG_ERR_CUDA;
    // persistent CTAs (two or one per SM by D), fewer when there is less work (the device knows
    // exactly how much)
    const int64_t work_bound = (int64_t)n_seq * max_q_tiles * Hq;
    auto launch = [&](auto kern, size_t smem, int per_sm) -> dg_status {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return DG_ERR_CUDA;
        const unsigned grid = (unsigned)std::max<int64_t>(1, std::min<int64_t>((int64_t)per_sm * P, work_bound));
        kern<<<grid, kThreads, smem, st>>>(tq, tk, tv, a, plan);
        dghost::count_launch();
        return dghost::cuda_status(cudaGetLastError());
    };
    if (D == 64) return launch(k_attention<64>, AttnCfg<64>::kSmem, AttnCfg<64>::kCtasPerSm);
    if (D == 128) return launch(k_attention<128>, AttnCfg<128>::kSmem, AttnCfg<128>::kCtasPerSm);
    return launch(k_attention<256>, AttnCfg<256>::kSmem, AttnCfg<256>::kCtasPerSm);
}
