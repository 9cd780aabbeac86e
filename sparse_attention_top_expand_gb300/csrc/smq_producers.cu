// Producers of the indexer's inputs on the GPU (sm_103a):
//   write_k_cache_kernel  bf16 keys -> the paged MXFP4 K cache (E2M1 values,
//                         one UE8M0 scale per 32 elements), through a slot
//                         mapping
//   quantize_q_kernel     bf16 query rows -> E4M3 codes and one float scale
//                         per row; float head weights -> bf16
// Rounding (the pages fix the formats, not the rounding):
//  - K: per group of 32, the smallest exponent e with amax <= 6 * 2^e (the
//    UE8M0 code e + 127, clamped to [1, 254]); elements x * 2^-e rounded to
//    the nearest E2M1 value, ties to even, saturating at 6.
//  - Q: scale = amax / 448 (1 for a zero row); elements x / scale (IEEE
//    float division) rounded to the nearest E4M3 value, ties to even,
//    saturating at 448. Weights: nearest-even bf16.
// Both kernels are bandwidth bound; inputs must be finite.
#include "smq_kernels.cuh"
#include "smq_ptx.cuh"

#include <cuda_bf16.h>

namespace smq {

namespace {

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// Two floats to two E2M1 codes in one byte: `lo` in the low nibble.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint32_t out;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u32.u8 %0, t;\n}" : "=r"(out) : "f"(hi), "f"(lo));
  return out;
}

// Two floats to two E4M3 codes in 16 bits: `lo` in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t out;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(out) : "f"(hi), "f"(lo));
  return out;
}

}  // namespace

// One warp per token: lane l holds elements 4l .. 4l + 3 (group l / 8).
__global__ void __launch_bounds__(256) write_k_cache_kernel(const __grid_constant__ KWriteParams p) {
  griddep_launch_dependents();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (t >= p.ntok) return;
  const int64_t slot = p.slot_mapping[t];
  if (slot < 0) return;  // a padding token
  const int64_t page = slot / p.page_size, off = slot % p.page_size;
  if (page >= p.num_pages) {
    if (lane == 0) atomicOr(p.status, kStatusBounds);
    return;
  }
  const uint2 raw = reinterpret_cast<const uint2*>(p.k + t * kHeadDim)[lane];
  float x[4] = {bf16_bits_to_f32(raw.x & 0xffffu), bf16_bits_to_f32(raw.x >> 16), bf16_bits_to_f32(raw.y & 0xffffu),
                bf16_bits_to_f32(raw.y >> 16)};
  float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
  for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));  // within 8 lanes
  // smallest e with amax <= 6 * 2^e: amax = m * 2^ex with m in [0.5, 1), so
  // e = ex - 3 if m <= 0.75, else ex - 2
  int code = 127;
  if (amax > 0.f) {
    int ex;
    const float m = frexpf(amax, &ex);
    code = (m <= 0.75f ? ex - 3 : ex - 2) + 127;
    code = code < 1 ? 1 : (code > 254 ? 254 : code);
  }
  const int e = code - 127;
  const uint32_t packed = e2m1x2(ldexpf(x[0], -e), ldexpf(x[1], -e)) |
                          (e2m1x2(ldexpf(x[2], -e), ldexpf(x[3], -e)) << 8);
  uint8_t* base = p.k_cache + page * p.page_bytes;
  reinterpret_cast<uint16_t*>(base + off * (kHeadDim / 2))[lane] = static_cast<uint16_t>(packed);
  const uint32_t c1 = __shfl_sync(0xffffffffu, code, 8), c2 = __shfl_sync(0xffffffffu, code, 16),
                 c3 = __shfl_sync(0xffffffffu, code, 24);
  if (lane == 0)
    *reinterpret_cast<uint32_t*>(base + static_cast<int64_t>(p.page_size) * (kHeadDim / 2) + off * kScaleWordBytes) =
        static_cast<uint32_t>(code) | (c1 << 8) | (c2 << 16) | (c3 << 24);
}

// One CTA of 256 threads per row of H x D elements.
__global__ void __launch_bounds__(256) quantize_q_kernel(const __grid_constant__ QQuantParams p) {
  griddep_launch_dependents();
  griddep_wait();
  __shared__ float red[8];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t r = blockIdx.x;
  const int n = p.heads * kHeadDim;
  const uint4* src = reinterpret_cast<const uint4*>(p.q + r * n);  // 8 bf16 per uint4
  float amax = 0.f;
  for (int i = tid; i < n / 8; i += 256) {
    const uint4 v = src[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      amax = fmaxf(amax, fmaxf(fabsf(bf16_bits_to_f32(w[j] & 0xffffu)), fabsf(bf16_bits_to_f32(w[j] >> 16))));
  }
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) amax = fmaxf(amax, red[w]);
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  uint2* dst = reinterpret_cast<uint2*>(p.q_fp8 + r * n);  // 8 codes per uint2
  for (int i = tid; i < n / 8; i += 256) {
    const uint4 v = src[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t c[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      c[j] = e4m3x2(__fdiv_rn(bf16_bits_to_f32(w[j] & 0xffffu), scale), __fdiv_rn(bf16_bits_to_f32(w[j] >> 16), scale));
    dst[i] = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
  }
  if (tid == 0) p.q_scale[r] = scale;
  for (int h = tid; h < p.heads; h += 256)
    p.weights_out[r * p.heads + h] = __bfloat16_as_ushort(__float2bfloat16_rn(p.weights_in[r * p.heads + h]));
}

namespace {

// Launch with programmatic stream serialisation (the kernels wait for the
// previous grid before reading anything).
template <typename P>
cudaError_t launch_pdl(void (*kernel)(P), unsigned grid, cudaStream_t stream, const P& params) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, params);
}

}  // namespace

cudaError_t launch_write_k_cache(const KWriteParams& p, cudaStream_t stream) {
  return launch_pdl(write_k_cache_kernel, static_cast<unsigned>((p.ntok + 7) / 8), stream, p);
}

cudaError_t launch_quantize_q(const QQuantParams& p, cudaStream_t stream) {
  return launch_pdl(quantize_q_kernel, static_cast<unsigned>(p.rows), stream, p);
}

}  // namespace smq
