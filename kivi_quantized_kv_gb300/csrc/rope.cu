// rope.cu — the rotation tables of a cache of pre-RoPE keys (KV-cache
// quantization guide (pigeon), "KVQuant adds": keys quantized before the
// rotary embedding).  Written once into the arena's workspace when a handle
// opens over such a cache, by one small kernel in double precision.
//
// Layout (floats): [theta]  θ_i = base^(-2i/d) for i < d/2 as two floats,
// hi = fl(θ_i) and lo = fl(θ_i - hi), so that a θ_i can be reduced mod 2π in
// fp32 without losing the product's low bits; then [offsets] for every even
// pair i and token offset j < G inside a group, 0.5 (cos jθ_i, sin jθ_i,
// cos jθ_(i+1), sin jθ_(i+1)) at float4 index (i / 2) (G + 1) + j (a lane
// turns two adjacent pairs of one token with one 16-byte load; the extra
// column j = G is zero).  The factor 0.5 keeps rotated keys of the full fp16
// range inside fp16; the decode takes it back with its score scale.
#include "kivi_internal.cuh"

#include <math.h>

namespace kivi {

namespace {

__global__ void rope_table_kernel(float* tab, double log2_base, int d, int G) {
  const int h = d / 2;
  const int x = blockIdx.x * blockDim.x + threadIdx.x;
  if (x < h) {
    const double th = exp2(-(2.0 * x / d) * log2_base);
    const float hi = static_cast<float>(th);
    tab[2 * x] = hi;
    tab[2 * x + 1] = static_cast<float>(th - static_cast<double>(hi));
  }
  if (x < (h / 2) * (G + 1)) {
    const int p = x / (G + 1), j = x % (G + 1);
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (j < G) {
      const double a0 = static_cast<double>(j) * exp2(-(2.0 * (2 * p) / d) * log2_base);
      const double a1 = static_cast<double>(j) * exp2(-(2.0 * (2 * p + 1) / d) * log2_base);
      v = make_float4(static_cast<float>(0.5 * cos(a0)), static_cast<float>(0.5 * sin(a0)),
                      static_cast<float>(0.5 * cos(a1)), static_cast<float>(0.5 * sin(a1)));
    }
    reinterpret_cast<float4*>(tab + d)[x] = v;
  }
}

}  // namespace

int64_t rope_table_bytes(const Geo& g) {
  return g.rope_l2b != 0.0 ? 4 * static_cast<int64_t>(g.d) + 8 * static_cast<int64_t>(g.d / 2) * (g.G + 1) : 0;
}

cudaError_t launch_rope_table(const Geo& g, uint8_t* arena, cudaStream_t stream) {
  if (g.rope_l2b == 0.0) return cudaSuccess;
  const int n = (g.d / 2) * (g.G + 1);
  if (injected_launch_failure()) return cudaErrorLaunchFailure;
  rope_table_kernel<<<(n + 255) / 256, 256, 0, stream>>>(reinterpret_cast<float*>(arena + g.ws_rope), g.rope_l2b,
                                                       g.d, g.G);
  return cudaGetLastError();
}

}  // namespace kivi
