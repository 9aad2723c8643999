// Weight repacking: checkpoint (output-major) 4-bit down projection ->
// neuron-major rows, and (scale, bias) interleaving.
//
// "Skipping dead neurons..." (sevren.ai), sections "Transposing to skip the
// zeros" and "Two layouts, one problem": decode needs the down weights one row
// per neuron so that a dead neuron's row is skipped in one piece; the
// checkpoint stores one row per output.  The numbers are the same.
#include "hs_common.cuh"

namespace hs {

// One CTA transposes a 64-output x 64-neuron tile of nibbles.
//   in : codes_om [out_dim][neurons/2]  (neuron 2j in the low nibble of byte j)
//   out: codes_nm [neurons][out_dim/2]  (output 2j in the low nibble of byte j)
__global__ void __launch_bounds__(256) repack_codes_kernel(const uint8_t* __restrict__ om, int out_dim,
                                                           int neurons, uint8_t* __restrict__ nm) {
    __shared__ uint8_t tile[64][65];  // [output][neuron] codes, padded
    const int o0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
    const int t = threadIdx.x;
    // load 64 rows x 32 bytes
    for (int i = t; i < 64 * 32; i += 256) {
        const int r = i >> 5, b = i & 31;
        const uint8_t v = om[(size_t)(o0 + r) * (neurons / 2) + n0 / 2 + b];
        tile[r][2 * b] = v & 15;
        tile[r][2 * b + 1] = v >> 4;
    }
    __syncthreads();
    for (int i = t; i < 64 * 32; i += 256) {
        const int n = i >> 5, b = i & 31;
        const uint8_t v = (uint8_t)(tile[2 * b][n] | (tile[2 * b + 1][n] << 4));
        nm[(size_t)(n0 + n) * (out_dim / 2) + o0 / 2 + b] = v;
    }
}

// sb_nm[g][o] = (scale_om[o][g], bias_om[o][g])
__global__ void repack_sb_kernel(const uint16_t* __restrict__ s, const uint16_t* __restrict__ b, int out_dim,
                                 int groups, uint32_t* __restrict__ sb) {
    const int o = blockIdx.x * blockDim.x + threadIdx.x;
    const int g = blockIdx.y;
    if (o >= out_dim) return;
    const size_t src = (size_t)o * groups + g;
    sb[(size_t)g * out_dim + o] = (uint32_t)s[src] | ((uint32_t)b[src] << 16);
}

// sb[i] = (scale[i], bias[i]) for a [rows][groups] pair of arrays
__global__ void pack_sb_kernel(const uint16_t* __restrict__ s, const uint16_t* __restrict__ b, size_t n,
                               uint32_t* __restrict__ sb) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) sb[i] = (uint32_t)s[i] | ((uint32_t)b[i] << 16);
}

// Re-quantisation of a checkpoint down projection with its scales along the
// neuron axis (section "The whole decode step": the checkpoint's scales per
// group of 64 neurons make one live neuron cost its group's scales).  Thread
// (n, j) takes neuron n's outputs 64j .. 64j+63: w = fma(s, q, b) in fp32
// (the exact value rounded once), scale = fp16((max - min) / 15), bias =
// fp16(min), q = clamp(rint((w - bias) / scale), 0, 15) (0 where scale is 0),
// every step rounded to fp32 as written.  Writes the neuron-major codes and
// the row's (scale, bias) pair for group j; thread (n, 0) zeroes the row's
// padding words.
__global__ void __launch_bounds__(256) requant_rowscale_kernel(const uint8_t* __restrict__ om,
                                                               const uint16_t* __restrict__ s_om,
                                                               const uint16_t* __restrict__ b_om, int out_dim,
                                                               int neurons, uint8_t* __restrict__ nm,
                                                               uint32_t* __restrict__ sb_row, int sbw) {
    const int n = blockIdx.x * blockDim.x + threadIdx.x, j = blockIdx.y;
    if (n >= neurons) return;
    const int Gn = neurons / 64;
    float w[64];
    float mx = -INFINITY, mn = INFINITY;
#pragma unroll
    for (int k = 0; k < 64; ++k) {
        const int o = 64 * j + k;
        const uint8_t byte = om[(size_t)o * (neurons / 2) + n / 2];
        const float q = (float)((n & 1) ? byte >> 4 : byte & 15);
        const size_t gi = (size_t)o * Gn + n / 64;
        w[k] = fmaf(__half2float(__ushort_as_half(s_om[gi])), q, __half2float(__ushort_as_half(b_om[gi])));
        mx = fmaxf(mx, w[k]);
        mn = fminf(mn, w[k]);
    }
    const __half sh = __float2half_rn((mx - mn) / 15.0f);
    const __half bh = __float2half_rn(mn);
    const float sf = __half2float(sh), bf = __half2float(bh);
    uint32_t packed[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t v = 0;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            const float qf = sf == 0.f ? 0.f : fminf(fmaxf(rintf((w[8 * i + m] - bf) / sf), 0.f), 15.f);
            v |= (uint32_t)qf << (4 * m);
        }
        packed[i] = v;
    }
    uint4* dst = reinterpret_cast<uint4*>(nm + (size_t)n * (out_dim / 2) + 32 * j);
    dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    uint32_t* row = sb_row + (size_t)n * sbw;
    row[j] = (uint32_t)__half_as_ushort(sh) | ((uint32_t)__half_as_ushort(bh) << 16);
    if (j == 0)
        for (int p = out_dim / 64; p < sbw; ++p) row[p] = 0u;
}

}  // namespace hs

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

extern "C" int hs_requant_down_rowscale(const uint8_t* codes_om, const uint16_t* scale_om, const uint16_t* bias_om,
                                        int out_dim, int neurons, uint8_t* codes_nm, void* sb_row,
                                        hs_stream_t stream) {
    if (!codes_om || !scale_om || !bias_om || !codes_nm || !sb_row) return HS_ERR_INVALID_ARG;
    if (out_dim <= 0 || neurons <= 0) return HS_ERR_INVALID_ARG;
    if (out_dim % 64 || neurons % 64) return HS_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(codes_nm) || !aligned16(sb_row) || ((uintptr_t)scale_om & 1) || ((uintptr_t)bias_om & 1))
        return HS_ERR_MISALIGNED;
    dim3 grid((neurons + 255) / 256, out_dim / 64);
    hs::requant_rowscale_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        codes_om, scale_om, bias_om, out_dim, neurons, codes_nm, reinterpret_cast<uint32_t*>(sb_row),
        hs_row_sb_words(out_dim));
    return cudaGetLastError() == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

extern "C" int hs_repack_down_nm(const uint8_t* codes_om, const uint16_t* scale_om, const uint16_t* bias_om,
                                 int out_dim, int neurons, uint8_t* codes_nm, void* sb_nm, hs_stream_t stream) {
    if (!codes_om || !scale_om || !bias_om || !codes_nm || !sb_nm) return HS_ERR_INVALID_ARG;
    if (out_dim <= 0 || neurons <= 0) return HS_ERR_INVALID_ARG;
    if (out_dim % 64 || neurons % 64) return HS_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(codes_om) || !aligned16(codes_nm) || !aligned16(sb_nm) || ((uintptr_t)scale_om & 1) ||
        ((uintptr_t)bias_om & 1))
        return HS_ERR_MISALIGNED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    dim3 g1(neurons / 64, out_dim / 64);
    hs::repack_codes_kernel<<<g1, 256, 0, s>>>(codes_om, out_dim, neurons, codes_nm);
    dim3 g2((out_dim + 255) / 256, neurons / 64);
    hs::repack_sb_kernel<<<g2, 256, 0, s>>>(scale_om, bias_om, out_dim, neurons / 64,
                                            reinterpret_cast<uint32_t*>(sb_nm));
    return cudaGetLastError() == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

extern "C" int hs_pack_sb(const uint16_t* scale, const uint16_t* bias, int rows, int groups, void* sb,
                          hs_stream_t stream) {
    if (!scale || !bias || !sb) return HS_ERR_INVALID_ARG;
    if (rows <= 0 || groups <= 0) return HS_ERR_INVALID_ARG;
    if (((uintptr_t)sb & 3) || ((uintptr_t)scale & 1) || ((uintptr_t)bias & 1)) return HS_ERR_MISALIGNED;
    const size_t n = (size_t)rows * groups;
    hs::pack_sb_kernel<<<(unsigned)((n + 255) / 256), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        scale, bias, n, reinterpret_cast<uint32_t*>(sb));
    return cudaGetLastError() == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}
