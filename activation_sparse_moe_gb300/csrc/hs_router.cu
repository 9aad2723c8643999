// Router projection of a MoE layer: one logit per routed expert and token,
// GB300 (sm_103a).
//
// "Skipping dead neurons..." (sevren.ai), section "Inside a MoE layer": a
// router picks 6 of 128 experts for each token.  The page does not print the
// router itself; it is read as the usual linear map from the token's hidden
// state to one logit per expert, logits[b][e] = sum_k W[e][k] x[b][k], with
// bf16 weights and activations and fp32 accumulation.  The top-6 and softmax
// that follow run inside the decode kernels.
//
// Design: one warp per expert row.  The warp keeps its row (hidden / 8
// 16-byte chunks, lane l holding chunks l, l + 32, ...) in registers, loaded
// before the wait for the previous kernel (the weights do not depend on it),
// and reuses it for every token; x comes through shared memory eight tokens
// at a time.  Each lane adds its products in chunk order into one fp32
// chain; the 32 lane sums are added by a fixed xor tree (deterministic).  A
// latency-bound GEMV (688 KB of weights per layer at hidden 2688); no tensor
// cores.
#include "hs_common.cuh"
#include "hs_host.h"

namespace hs {

constexpr int kRouterWarps = 8;                    // experts per CTA
constexpr int kRouterTok = 8;                      // tokens per x tile in shared memory
constexpr int kRouterChunks = kMaxHidden / 8 / 32; // 16-byte chunks per lane at the largest hidden size

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__global__ void __launch_bounds__(kRouterWarps * 32) router_logits_kernel(const uint16_t* __restrict__ x,
                                                                          const uint16_t* __restrict__ w, int B,
                                                                          int H, int E, float* __restrict__ logits) {
    extern __shared__ __align__(16) uint16_t xs[];  // [kRouterTok][H]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int e = blockIdx.x * kRouterWarps + warp;
    const int nch = H / 8;
    uint4 wr[kRouterChunks];
#pragma unroll
    for (int i = 0; i < kRouterChunks; ++i) {
        const int c = lane + 32 * i;
        wr[i] = (e < E && c < nch) ? __ldg(reinterpret_cast<const uint4*>(w + (size_t)e * H) + c)
                                   : make_uint4(0, 0, 0, 0);
    }
    pdl_wait();
    pdl_trigger();
    for (int b0 = 0; b0 < B; b0 += kRouterTok) {
        const int nb = min(kRouterTok, B - b0);
        __syncthreads();  // the previous tile is consumed
        for (int i = threadIdx.x; i < nb * nch; i += blockDim.x)
            reinterpret_cast<uint4*>(xs)[i] = __ldcg(reinterpret_cast<const uint4*>(x + (size_t)b0 * H) + i);
        __syncthreads();
        if (e >= E) continue;
        for (int j = 0; j < nb; ++j) {
            const uint4* xr = reinterpret_cast<const uint4*>(xs + (size_t)j * H);
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < kRouterChunks; ++i) {
                const int c = lane + 32 * i;
                if (c < nch) {
                    const uint4 xv = xr[c];
                    const uint32_t wv4[4] = {wr[i].x, wr[i].y, wr[i].z, wr[i].w};
                    const uint32_t xv4[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        acc = fmaf(bf16_lo(wv4[q]), bf16_lo(xv4[q]), acc);
                        acc = fmaf(bf16_hi(wv4[q]), bf16_hi(xv4[q]), acc);
                    }
                }
            }
#pragma unroll
            for (int off = 16; off; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (lane == 0) logits[(size_t)(b0 + j) * E + e] = acc;
        }
    }
}

}  // namespace hs

using namespace hs_host;

extern "C" int hs_router_logits(const uint16_t* x, const uint16_t* w_router, int batch, int hidden, int n_experts,
                                float* logits, hs_stream_t stream) {
    if (!x || !w_router || !logits) return HS_ERR_INVALID_ARG;
    if (batch < 1 || hidden < 1 || n_experts < 1) return HS_ERR_INVALID_ARG;
    if (hidden % 64 || hidden > hs::kMaxHidden) return HS_ERR_UNSUPPORTED_SHAPE;
    if (!al16(x) || !al16(w_router) || !al4(logits)) return HS_ERR_MISALIGNED;
    const int smem = std::min(batch, hs::kRouterTok) * hidden * 2;  // at most 48 KB
    if (launch_pdl(hs::router_logits_kernel, dim3((n_experts + hs::kRouterWarps - 1) / hs::kRouterWarps),
                   dim3(hs::kRouterWarps * 32), smem, reinterpret_cast<cudaStream_t>(stream), x, w_router, batch,
                   hidden, n_experts, logits) != cudaSuccess)
        return HS_ERR_CUDA;
    return launch_err();
}
