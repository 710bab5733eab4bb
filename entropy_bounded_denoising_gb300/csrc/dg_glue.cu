// dg_glue.cu -- around the denoise step: single-pass-read choice probabilities, the next
// pass's canvas embeddings (token embedding + stored feedback) and the commit of converged
// canvases.
//
// Method: single-pass reads page ("답은 한 번 읽는데 모델은 왜 두 번 돌까? DiffusionGemma의
// 실행 경로 합치기"), section "답의 내용은 몰라도 답을 담을 자리는 안다" (a read-only request
// reads the probabilities of fixed answer tokens at its answer slots); DiffusionGemma vLLM
// page ("DiffusionGemma: vLLM이 네이티브로 지원하는 최초의 디퓨전 언어 모델(dLLM)"), section
// "DiffusionGemmaModelState와 DiffusionSampler" (the input-preparation hook adds the stored
// feedback to the canvas embeddings; the Commit case emits the converged argmax canvas) and
// section "자기 조건화" (the feedback joins the next pass's canvas embeddings).
//
// All three are memory-bound gathers: one thread per output slot (choice probabilities),
// per 16-byte chunk of an embedding row (8 bf16 values, coalesced along the row), per
// canvas position (commit).
#include <cuda_runtime.h>

#include <math.h>

#include <algorithm>

#include "dg_common.cuh"

namespace {

__global__ void __launch_bounds__(256) k_choice_probs(const unsigned char* __restrict__ logits, int dt,
                                                      int64_t ld_bytes, const float* __restrict__ lse,
                                                      const dg_canvas_params* __restrict__ params, int32_t L,
                                                      int64_t V, const int32_t* __restrict__ choices, int32_t C,
                                                      float* __restrict__ probs, int64_t total, unsigned* status) {
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < total; q += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = q / C;          // canvas * L + position
        const int64_t c = row / L;
        const dg_canvas_params p = params[c];
        if (!(p.flags & DG_ACTIVE)) continue;
        if (!(p.temperature > 0.f) || !isfinite(p.temperature)) {
            if (q % ((int64_t)L * C) == 0) dg::raise_status(status, DG_DEV_BAD_PARAM);
            continue;
        }
        const int32_t tok = choices[q];
        float out = 0.f;
        if (tok >= 0 && (int64_t)tok < V) {
            const unsigned char* src = logits + row * ld_bytes;
            const float x = dt == 0 ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(src)[tok] << 16)
                                    : reinterpret_cast<const float*>(src)[tok];
            const float invT = 1.0f / p.temperature;  // the same scaling as the step's statistics
            out = expf(x * invT - lse[row]);
        }
        probs[q] = out;
    }
}

DG_DEVINL uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// One fp32 fma per element: scale * e + a, rounded to nearest even to bf16, for the 8
// entries of a 16-byte chunk.
DG_DEVINL uint32_t fma_pair(uint32_t e2, uint32_t a2, float scale) {
    const float e0 = __uint_as_float(e2 << 16), e1 = __uint_as_float(e2 & 0xffff0000u);
    const float a0 = __uint_as_float(a2 << 16), a1 = __uint_as_float(a2 & 0xffff0000u);
    return pack_bf16x2(fmaf(scale, e0, a0), fmaf(scale, e1, a1));
}

__global__ void __launch_bounds__(256) k_embed(const int32_t* __restrict__ canvas, int64_t n_rows, int64_t V,
                                               const uint16_t* __restrict__ E, int32_t d,
                                               const uint16_t* __restrict__ delta, float scale,
                                               uint16_t* __restrict__ out, unsigned* status) {
    const int64_t cpr = d / 8;  // 16-byte chunks per row
    const int64_t total = n_rows * cpr;
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < total; q += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = q / cpr, ch = q % cpr;
        const int32_t tok = canvas[r];
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (tok >= 0 && (int64_t)tok < V) {
            const uint4 e = *reinterpret_cast<const uint4*>(E + (int64_t)tok * d + ch * 8);
            const uint4 a = delta ? *reinterpret_cast<const uint4*>(delta + r * d + ch * 8) : make_uint4(0u, 0u, 0u, 0u);
            o = make_uint4(fma_pair(e.x, a.x, scale), fma_pair(e.y, a.y, scale), fma_pair(e.z, a.z, scale),
                           fma_pair(e.w, a.w, scale));
        } else if (ch == 0) {
            dg::raise_status(status, DG_DEV_BAD_PARAM);
        }
        *reinterpret_cast<uint4*>(out + r * d + ch * 8) = o;
    }
}

__global__ void __launch_bounds__(1024) k_commit(const dg_canvas_params* __restrict__ params,
                                                 const uint8_t* __restrict__ converged,
                                                 const int32_t* __restrict__ argmax, int32_t L,
                                                 int32_t* __restrict__ tokens, int32_t* __restrict__ prev_argmax,
                                                 int32_t* __restrict__ stable_count, uint8_t* __restrict__ committed) {
    const int64_t c = blockIdx.x;
    const int i = threadIdx.x;
    const bool go = (params[c].flags & DG_ACTIVE) && converged[c];
    if (i == 0) {
        committed[c] = go ? 1 : 0;
        if (go) stable_count[c] = 0;
    }
    if (!go || i >= L) return;
    const int64_t q = c * L + i;
    tokens[q] = argmax[q];
    prev_argmax[q] = -1;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

unsigned blocks_for(int64_t work, int per_block) {
    const int64_t want = (work + per_block - 1) / per_block;
    const int64_t cap = 8LL * std::max(1, dghost::sm_count()) * 8;  // a few waves, grid-stride beyond
    return (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, cap));
}

}  // namespace

extern "C" {

dg_status dg_choice_probs(const void* logits, dg_dtype dtype, int64_t ld, const float* lse,
                          const dg_canvas_params* params, int64_t n_canvas, int32_t L, int64_t V,
                          const int32_t* choices, int32_t C, float* probs, dg_stream_t stream) {
    if (dtype != DG_BF16 && dtype != DG_FP32) return DG_ERR_INVALID_ARG;
    if (n_canvas < 0 || n_canvas > 65535 || L < 1 || L > 1024 || V < 2 || V > 0x7fffffffLL || ld < V || C < 1 ||
        C > 1024)
        return DG_ERR_INVALID_ARG;
    if (n_canvas == 0) return DG_OK;
    if (!logits || !lse || !params || !choices || !probs) return DG_ERR_INVALID_ARG;
    if (!aligned16(logits)) return DG_ERR_ALIGNMENT;
    const int64_t es = dtype == DG_BF16 ? 2 : 4;
    const int64_t total = n_canvas * L * (int64_t)C;
    k_choice_probs<<<blocks_for(total, 256), 256, 0, (cudaStream_t)stream>>>(
        static_cast<const unsigned char*>(logits), dtype == DG_BF16 ? 0 : 1, ld * es, lse, params, L, V, choices, C,
        probs, total, dghost::status_word());
    dghost::count_launch();
    return dghost::cuda_status(cudaGetLastError());
}

dg_status dg_embed_canvas(const int32_t* canvas, int64_t n_rows, int64_t V, const uint16_t* E, int32_t d,
                          const uint16_t* delta_emb, float scale, uint16_t* out, dg_stream_t stream) {
    if (n_rows < 0 || n_rows > 0x7fffffffLL || V < 2 || V > 0x7fffffffLL || d < 8 || d > 65536 || (d % 8))
        return DG_ERR_INVALID_ARG;
    if (n_rows == 0) return DG_OK;
    if (!canvas || !E || !out) return DG_ERR_INVALID_ARG;
    if (!aligned16(E) || !aligned16(out) || (delta_emb && !aligned16(delta_emb))) return DG_ERR_ALIGNMENT;
    const int64_t work = n_rows * (d / 8);
    k_embed<<<blocks_for(work, 256), 256, 0, (cudaStream_t)stream>>>(canvas, n_rows, V, E, d, delta_emb, scale, out,
                                                                     dghost::status_word());
    dghost::count_launch();
    return dghost::cuda_status(cudaGetLastError());
}

dg_status dg_commit(const dg_canvas_params* params, const uint8_t* converged, const int32_t* argmax,
                    int64_t n_canvas, int32_t L, int32_t* tokens, int32_t* prev_argmax, int32_t* stable_count,
                    uint8_t* committed, dg_stream_t stream) {
    if (n_canvas < 0 || n_canvas > 65535 || L < 1 || L > 1024) return DG_ERR_INVALID_ARG;
    if (n_canvas == 0) return DG_OK;
    if (!params || !converged || !argmax || !tokens || !prev_argmax || !stable_count || !committed)
        return DG_ERR_INVALID_ARG;
    const unsigned threads = (unsigned)((L + 31) / 32 * 32);
    k_commit<<<(unsigned)n_canvas, threads, 0, (cudaStream_t)stream>>>(params, converged, argmax, L, tokens,
                                                                       prev_argmax, stable_count, committed);
    dghost::count_launch();
    return dghost::cuda_status(cudaGetLastError());
}

}  // extern "C"
