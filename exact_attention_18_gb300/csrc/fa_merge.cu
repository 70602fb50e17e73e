// Split-KV merge: attention over a key set split into shards, each shard's
// normalised partial output O_s and logsumexp L_s already computed, combined
// exactly into the full result ("T5 讲解" §⑥: storing L = m + log l is what
// lets shards be merged):
//
//   L = ln sum_s exp(L_s),   O = sum_s exp(L_s - L) O_s.
//
// Each O_s is a softmax-weighted mean over the shard's keys, and exp(L_s - L)
// is the shard's share of the row's total softmax mass, so the sum is the
// softmax over all keys.  A shard in which the row sees no key has L_s = -inf
// and weight 0; a row that sees no key at all gets O = 0, L = -inf.  The
// kernel is bound by HBM: it reads every partial once.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa_kernel_common.cuh"

namespace fa {

namespace {

// One thread per 8 columns of a row (D/8 threads per row), grid-stride over
// rows.  o_part: [shards][rows][D] fp32; lse_part: [shards][rows] fp32.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_merge_lse_kernel(const float* __restrict__ o_part,
                                                           const float* __restrict__ lse_part, int shards,
                                                           int64_t rows, void* __restrict__ o, float* __restrict__ lse) {
  constexpr int kTpr = D / 8;  // threads per row
  const int64_t n = rows * kTpr;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = e / kTpr;
    const int cg = static_cast<int>(e - row * kTpr);
    float mx = -INFINITY;
    for (int s = 0; s < shards; ++s) mx = fmaxf(mx, __ldg(lse_part + s * rows + row));
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float total = 0.f;
    if (mx != -INFINITY) {
      for (int s = 0; s < shards; ++s) {
        const float w = expf(__ldg(lse_part + s * rows + row) - mx);  // 0 for a shard with L_s = -inf
        total += w;
        const float4* src = reinterpret_cast<const float4*>(o_part + (s * rows + row) * D + cg * 8);
        const float4 a = __ldg(src), b = __ldg(src + 1);
        acc[0] += w * a.x; acc[1] += w * a.y; acc[2] += w * a.z; acc[3] += w * a.w;
        acc[4] += w * b.x; acc[5] += w * b.y; acc[6] += w * b.z; acc[7] += w * b.w;
      }
    }
    const float inv = total > 0.f ? 1.f / total : 0.f;
    const uint4 out = make_uint4(pack2<BF16>(acc[0] * inv, acc[1] * inv), pack2<BF16>(acc[2] * inv, acc[3] * inv),
                                 pack2<BF16>(acc[4] * inv, acc[5] * inv), pack2<BF16>(acc[6] * inv, acc[7] * inv));
    reinterpret_cast<uint4*>(static_cast<char*>(o) + (row * D + cg * 8) * 2)[0] = out;
    if (cg == 0) lse[row] = total > 0.f ? mx + logf(total) : -INFINITY;
  }
}

template <int D, bool BF16>
cudaError_t launch_merge_t(const float* o_part, const float* lse_part, int shards, int64_t rows, void* o, float* lse,
                           cudaStream_t stream) {
  const int64_t threads = rows * (D / 8);
  const int64_t blocks = (threads + 255) / 256;
  const int grid = static_cast<int>(blocks < 152 * 16 ? blocks : 152 * 16);
  fa_merge_lse_kernel<D, BF16><<<grid, 256, 0, stream>>>(o_part, lse_part, shards, rows, o, lse);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_merge_lse(int D, bool bf16, const float* o_part, const float* lse_part, int shards, int64_t rows,
                             void* o, float* lse, cudaStream_t stream) {
  switch (D) {
    case 16: return bf16 ? launch_merge_t<16, true>(o_part, lse_part, shards, rows, o, lse, stream)
                         : launch_merge_t<16, false>(o_part, lse_part, shards, rows, o, lse, stream);
    case 32: return bf16 ? launch_merge_t<32, true>(o_part, lse_part, shards, rows, o, lse, stream)
                         : launch_merge_t<32, false>(o_part, lse_part, shards, rows, o, lse, stream);
    case 64: return bf16 ? launch_merge_t<64, true>(o_part, lse_part, shards, rows, o, lse, stream)
                         : launch_merge_t<64, false>(o_part, lse_part, shards, rows, o, lse, stream);
    case 128: return bf16 ? launch_merge_t<128, true>(o_part, lse_part, shards, rows, o, lse, stream)
                          : launch_merge_t<128, false>(o_part, lse_part, shards, rows, o, lse, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fa
