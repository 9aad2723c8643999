// Host-side helpers shared by the libhs translation units: argument checks,
// launches with programmatic dependent launch, kernel attribute setup.
#pragma once

#include <cuda_runtime.h>
#include <cstring>
#include <mutex>

#include "hs.h"
#include "hs_kernels.cuh"

namespace hs_host {

inline bool al16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
inline bool al4(const void* p) { return ((uintptr_t)p & 3u) == 0; }

inline size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline int launch_err() { return cudaGetLastError() == cudaSuccess ? HS_OK : HS_ERR_CUDA; }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Raises a kernel's dynamic shared memory limit once per (kernel, device, size):
// the attribute call is kept out of the per-call path (and out of stream capture
// after the first eager call).
inline int set_smem_attr(const void* fn, int bytes) {
    struct Entry { const void* fn; int dev; int bytes; };
    static Entry done[64];
    static int n_done = 0;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return HS_ERR_CUDA;
    for (int i = 0; i < n_done; ++i)
        if (done[i].fn == fn && done[i].dev == dev && done[i].bytes >= bytes) return HS_OK;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return HS_ERR_CUDA;
    if (n_done < 64) done[n_done++] = Entry{fn, dev, bytes};
    return HS_OK;
}

inline int check_expert(const hs_expert& e, int hidden, int neurons_expected) {
    if (!e.up.codes || !e.up.sb || !e.down_nm.codes || !e.down_nm.sb) return HS_ERR_INVALID_ARG;
    if (e.neurons != neurons_expected) return HS_ERR_UNSUPPORTED_SHAPE;
    if (!al16(e.up.codes) || !al16(e.up.sb) || !al16(e.down_nm.codes) || !al16(e.down_nm.sb)) return HS_ERR_MISALIGNED;
    if (e.up_offset && !al4(e.up_offset)) return HS_ERR_MISALIGNED;
    (void)hidden;
    return HS_OK;
}

// The reduce pass holds one 128-byte row per unit in shared memory.
constexpr int kMaxUnits = 1536;

inline int check_layer(const hs_moe_layer* L) {
    if (!L || !L->routed) return HS_ERR_INVALID_ARG;
    if (L->n_routed < 1 || L->n_routed > hs::kMaxRouted) return HS_ERR_UNSUPPORTED_SHAPE;
    if (L->top_k < 1 || L->top_k > hs::kMaxTopK || L->top_k > L->n_routed) return HS_ERR_UNSUPPORTED_SHAPE;
    if (L->hidden < 64 || L->hidden > hs::kMaxHidden || L->hidden % 64) return HS_ERR_UNSUPPORTED_SHAPE;
    const int rn = L->routed[0].neurons;
    if (rn < 64 || rn % 64) return HS_ERR_UNSUPPORTED_SHAPE;
    for (int e = 0; e < L->n_routed; ++e) {
        const int st = check_expert(L->routed[e], L->hidden, rn);
        if (st != HS_OK) return st;
    }
    if (L->shared) {
        if (L->shared->neurons < 64 || L->shared->neurons % 64) return HS_ERR_UNSUPPORTED_SHAPE;
        const int st = check_expert(*L->shared, L->hidden, L->shared->neurons);
        if (st != HS_OK) return st;
    }
    if ((L->shared ? L->shared->neurons / 64 : 0) + L->top_k * (rn / 64) > kMaxUnits) return HS_ERR_UNSUPPORTED_SHAPE;
    return HS_OK;
}

inline int decode_units(const hs_moe_layer* L) {
    return (L->shared ? L->shared->neurons / 64 : 0) + L->top_k * (L->routed[0].neurons / 64);
}


// Kernel-parameter copy of a layer descriptor (pointers, uniform strides).
inline void fill_layer_params(const hs_moe_layer* L, hs::LayerParams& P) {
    memset(&P, 0, sizeof(P));
    auto fill = [](hs::ExpertPtrs& d, const hs_expert& e) {
        d.up_codes = e.up.codes;
        d.up_sb = static_cast<const uint32_t*>(e.up.sb);
        d.dn_codes = e.down_nm.codes;
        d.dn_sb = static_cast<const uint32_t*>(e.down_nm.sb);
        d.up_off = e.up_offset;
    };
    for (int e = 0; e < L->n_routed; ++e) fill(P.routed[e], L->routed[e]);
    if (L->shared) fill(P.shared, *L->shared);
    auto fld = [&](int e, int f) -> long long {
        const hs::ExpertPtrs& d = P.routed[e];
        const void* v[5] = {d.up_codes, d.up_sb, d.dn_codes, d.dn_sb, d.up_off};
        return (long long)(uintptr_t)v[f];
    };
    bool uni = true;
    for (int f = 0; f < 5; ++f) {
        const long long st = L->n_routed > 1 ? fld(1, f) - fld(0, f) : 0;
        P.stride[f] = st;
        for (int e = 0; e < L->n_routed && uni; ++e) uni = (fld(e, f) == fld(0, f) + e * st);
        if (f == 4)
            for (int e = 0; e < L->n_routed && uni; ++e) uni = ((fld(e, 4) == 0) == (fld(0, 4) == 0));
    }
    P.uniform = uni ? 1 : 0;
    P.n_routed = L->n_routed;
    P.routed_neurons = L->routed[0].neurons;
    P.shared_neurons = L->shared ? L->shared->neurons : 0;
    P.hidden = L->hidden;
    P.top_k = L->top_k;
}

}  // namespace hs_host

// Batch (> 1 token) decode, in hs_batch.cu.
size_t hs_batch_decode_workspace_size(const hs_moe_layer* L, int batch);
int hs_batch_decode(const hs_moe_layer* L, const uint16_t* x, const float* logits, int batch, uint16_t* y_bf16,
                    float* y_f32, unsigned flags, const hs_decode_debug* dbg, void* ws, size_t ws_bytes,
                    cudaStream_t stream);
// Reads and clears the batch translation unit's device error word.
unsigned hs_batch_take_status();
// Reads and clears the prefill translation unit's device error word.
unsigned hs_prefill_take_status();
// Batch decode of this many tokens or more runs on the prefill kernels (tensor
// cores: each weight tile is dequantised once for all of an expert's tokens),
// where the layer allows it; below, the batch decode kernels are faster.
constexpr int kPrefillMinBatch = 51;
// HS_OK if hs_moe_prefill takes this layer and token count.
int hs_prefill_layer_ok(const hs_moe_layer* L, int tokens);
// After an hs_moe_prefill call on workspace ws (stream-ordered): the union
// over each expert's tokens of its live neurons (h > 0), summed over the
// experts, and the 64-neuron groups holding one.  Either output may be null.
int hs_prefill_union_live(const hs_moe_layer* L, int tokens, void* ws, int* live_rows, int* live_groups,
                          cudaStream_t stream);
