// Per-row softmax pieces shared by the forward kernels: the scaled block
// maximum and the exponentials of one key block for a thread that owns one
// query row (TMEM lane), in the base-2 domain of "fa-triton" Step 2
// (c = scale * log2 e folded into one multiply-add).
#pragma once

#include "fa_kernel_common.cuh"

namespace fa {

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float min3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Scaled row maximum c * max_k s_k over the NC scores of a block (the minimum
// raw score when c < 0, whose scaled value is then the largest); with
// `masked`, only columns k <= lim (and, with LO, k >= lo) count.  -inf if no
// column is visible.
template <int NC, bool LO = false>
__device__ __forceinline__ float block_max_scaled(const uint32_t* sr, bool masked, int lo, int lim, float sl2,
                                                  bool neg) {
  static_assert(NC % 16 == 0, "block width");
  float mx;
  if (!masked) {
    // NC/16 independent chains of 3-input max/min keep the dependency depth short.
    constexpr int kChains = NC / 16;
    float mc[kChains];
#pragma unroll
    for (int k = 0; k < kChains; ++k) {
      const uint32_t* v = sr + 16 * k;
      float a = neg ? min3(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]))
                    : max3(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]));
#pragma unroll
      for (int c = 3; c < 15; c += 2)
        a = neg ? min3(a, __uint_as_float(v[c]), __uint_as_float(v[c + 1]))
                : max3(a, __uint_as_float(v[c]), __uint_as_float(v[c + 1]));
      mc[k] = neg ? fminf(a, __uint_as_float(v[15])) : fmaxf(a, __uint_as_float(v[15]));
    }
    mx = mc[0];
#pragma unroll
    for (int k = 1; k < kChains; ++k) mx = neg ? fminf(mx, mc[k]) : fmaxf(mx, mc[k]);
  } else {
    mx = neg ? INFINITY : -INFINITY;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const float x = __uint_as_float(sr[c]);
      if (c <= lim && (!LO || c >= lo)) mx = neg ? fminf(mx, x) : fmaxf(mx, x);
    }
  }
  if constexpr (LO) {
    if (masked && (lo > NC - 1 || lim < lo)) return -INFINITY;
  }
  return lim < 0 ? -INFINITY : mx * sl2;
}

// P~_k = exp2(c * s_k - m) for scores k0 .. k0+15 of a block, packed as eight
// 16-bit pairs into pk (key k0+2i in the low half of pk[i]); with MASKED,
// columns past lim (and, with LO, before lo) are exactly 0.  The unrounded P~
// are added into acc.  MASKED is a template parameter so the unmasked blocks
// (all but the diagonal and ragged ones) carry no per-element compare or select.
template <bool BF16, bool MASKED, bool LO = false>
__device__ __forceinline__ void exp16(const uint32_t* sr, int k0, float2 c2, float2 negm, int lo, int lim,
                                      float2* acc, uint32_t* pk) {
#pragma unroll
  for (int c = 0; c < 16; c += 2) {
    const float2 y =
        __ffma2_rn(make_float2(__uint_as_float(sr[k0 + c]), __uint_as_float(sr[k0 + c + 1])), c2, negm);
    float2 e = make_float2(ptx::ex2(y.x), ptx::ex2(y.y));
    if constexpr (MASKED) {
      if (k0 + c > lim || (LO && k0 + c < lo)) e.x = 0.f;
      if (k0 + c + 1 > lim || (LO && k0 + c + 1 < lo)) e.y = 0.f;
    }
    acc[(c / 2) & 3] = __fadd2_rn(acc[(c / 2) & 3], e);
    pk[c / 2] = pack2<BF16>(e.x, e.y);
  }
}

// Warp-collective: after this warp's tcgen05 stores/loads are complete, one
// elected lane arrives on `bar` (whose count is the number of arriving warps).
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
  ptx::tc_fence_before();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(bar);
}

}  // namespace fa
