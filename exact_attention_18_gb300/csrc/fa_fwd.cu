// Forward kernel: exact attention with an online softmax, FlashAttention-2
// loop order (query block outer, key/value block inner), on tcgen05 tensor
// cores with accumulators in tensor memory (TMEM).
//
// One CTA per (batch*head, 128-row query tile).  Warp roles:
//   warps 0-3  softmax / correction / epilogue; thread t owns query row t,
//              which is TMEM lane t (each thread holds whole rows, so row
//              max and row sum need no cross-thread reduction — the split-Q
//              work partition of "Inside FlashAttention" §4.3);
//   warp 4     TMA producer: Q once, then K and V blocks through a ring of
//              shared-memory stages;
//   warp 5     MMA issuer: S = Q K^T into TMEM, then O += P V with P read
//              from TMEM (written there by the softmax warps over S).
//
// Per key block j, for each row (base-2 domain, c = scale * log2 e):
//   m_new = max(m_old, c * rowmax(S_j))           ("T5 讲解" §④; "fa-triton" Step 2)
//   P~    = exp2(c * S_j - m_new)                 (exp2 with log2 e folded in, "fa-triton" Step 3)
//   l     = alpha * l + rowsum(P~),  alpha = exp2(m_old - m_new)
//   O     = alpha * O + P~ V                       (deferred 1/l, "Inside FlashAttention" §4.1)
// O is rescaled only for warps in which some row's maximum moved; when it
// did not, alpha is exactly 1.  Epilogue: O / l and L = (m + log2 l) * ln 2.
//
// Causal: query tile m visits key blocks 0..m only ("T5 讲解" §⑤); the mask
// is applied element-wise only in the diagonal block and in a ragged last
// key block ("fa-triton" §Causal Mask 的处理：off-band 与 on-band).
#include "fa_kernel_common.cuh"

namespace fa {
using namespace ptx;

namespace {

template <int D>
struct FwdLayout : TileGeom<D> {
  using G = TileGeom<D>;
  static constexpr int kStages = D <= 64 ? 3 : 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + G::kTileBytes;
  static constexpr int kOffV = kOffK + kStages * G::kTileBytes;
  static constexpr int kOffBar = kOffV + kStages * G::kTileBytes;
  // q, kfull[S], vfull[S], empty[S], sfull[2], pfull[2], pvdone[2], drain
  static constexpr int kNumBars = 1 + 3 * kStages + 6 + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemUsed = kOffMisc + 16;
  // Tensor memory is allocated whole (512 columns), so at most one CTA may
  // live on an SM: the request is padded above half of the SM's shared memory.
  static constexpr int kSmemBytes = (kSmemUsed + 1024) > 116 * 1024 ? (kSmemUsed + 1024) : 116 * 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 256;  // S buffers at columns 0 and 128
};

}  // namespace

template <int D, bool BF16>
__global__ void __launch_bounds__(192, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using L = FwdLayout<D>;
  using elem_t = typename std::conditional<BF16, __nv_bfloat16, __half>::type;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* bar_q = bars;
  uint64_t* bar_kfull = bars + 1;
  uint64_t* bar_vfull = bar_kfull + L::kStages;
  uint64_t* bar_empty = bar_vfull + L::kStages;
  uint64_t* bar_sfull = bar_empty + L::kStages;
  uint64_t* bar_pfull = bar_sfull + 2;
  uint64_t* bar_pvdone = bar_pfull + 2;
  uint64_t* bar_drain = bar_pvdone + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int S = p.S;
  const int m_tile = p.causal ? (p.n_m_tiles - 1 - static_cast<int>(blockIdx.y)) : static_cast<int>(blockIdx.y);
  const int row0 = m_tile * kBlockM;
  const int n_kv = (S + kBlockN - 1) / kBlockN;
  const int nblk = p.causal ? min(n_kv, (row0 + kBlockM + kBlockN - 1) / kBlockN) : n_kv;

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(&bar_kfull[s], 1);
      mbar_init(&bar_vfull[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_sfull[b], 1);
      mbar_init(&bar_pfull[b], 128);
      mbar_init(&bar_pvdone[b], 1);
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const uint32_t sQ = smem_u32(smem + L::kOffQ);
  const uint32_t sK = smem_u32(smem + L::kOffK);
  const uint32_t sV = smem_u32(smem + L::kOffV);

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      mbar_arrive_expect_tx(bar_q, L::kTileBytes);
#pragma unroll
      for (int ch = 0; ch < L::kChunks; ++ch)
        tma_load_3d(smem + L::kOffQ + ch * L::kChunkBytes, &tm_q, bar_q, ch * (L::kRowBytes / 2), row0, bh);
      int it = 0;
      for (; it < nblk; ++it) {
        const int st = it % L::kStages;
        const int use = it / L::kStages;
        if (use > 0 && !mbar_wait(&bar_empty[st], (use - 1) & 1, abort_flag, p.err, kErrTimeoutLoad)) break;
        mbar_arrive_expect_tx(&bar_kfull[st], L::kTileBytes);
#pragma unroll
        for (int ch = 0; ch < L::kChunks; ++ch)
          tma_load_3d(smem + L::kOffK + st * L::kTileBytes + ch * L::kChunkBytes, &tm_k, &bar_kfull[st],
                      ch * (L::kRowBytes / 2), it * kBlockN, bh);
        mbar_arrive_expect_tx(&bar_vfull[st], L::kTileBytes);
#pragma unroll
        for (int ch = 0; ch < L::kChunks; ++ch)
          tma_load_3d(smem + L::kOffV + st * L::kTileBytes + ch * L::kChunkBytes, &tm_v, &bar_vfull[st],
                      ch * (L::kRowBytes / 2), it * kBlockN, bh);
      }
      // Teardown: every copy this thread started must land before the CTA exits.
      drain_wait(bar_q, 0, p.err);
      for (int x = (it > L::kStages ? it - L::kStages : 0); x < it; ++x) {
        const int st = x % L::kStages;
        drain_wait(&bar_kfull[st], (x / L::kStages) & 1, p.err);
        drain_wait(&bar_vfull[st], (x / L::kStages) & 1, p.err);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = make_idesc_f16(BF16, 128, kBlockN, false, false);
      constexpr uint32_t idesc_pv = make_idesc_f16(BF16, 128, D, false, true);
      const uint32_t t_o = tmem + L::kColO;
      auto issue_pv = [&](int x) -> bool {
        const int b = x & 1;
        const int st = x % L::kStages;
        if (!mbar_wait(&bar_pfull[b], (x >> 1) & 1, abort_flag, p.err, kErrTimeoutMma)) return false;
        if (!mbar_wait(&bar_vfull[st], (x / L::kStages) & 1, abort_flag, p.err, kErrTimeoutMma)) return false;
        tc_fence_after();
        const uint32_t t_p = tmem + 128u * b;
        const uint32_t v_addr = sV + st * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk)
          mma_ts(t_o, t_p + kk * 8, mnmajor_desc<D>(v_addr, kk), idesc_pv, (x > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bar_pvdone[b]);
        mma_commit(&bar_empty[st]);
        return true;
      };
      bool ok = mbar_wait(bar_q, 0, abort_flag, p.err, kErrTimeoutMma);
      for (int it = 0; ok && it < nblk; ++it) {
        const int st = it % L::kStages;
        const int b = it & 1;
        ok = mbar_wait(&bar_kfull[st], (it / L::kStages) & 1, abort_flag, p.err, kErrTimeoutMma);
        if (ok && it >= 2) ok = mbar_wait(&bar_pvdone[b], ((it - 2) >> 1) & 1, abort_flag, p.err, kErrTimeoutMma);
        if (!ok) break;
        tc_fence_after();
        const uint32_t t_s = tmem + 128u * b;
        const uint32_t k_addr = sK + st * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(t_s, kmajor_desc<D>(sQ, kk), kmajor_desc<D>(k_addr, kk), idesc_qk, kk > 0 ? 1u : 0u);
        mma_commit(&bar_sfull[b]);
        if (it >= 1) ok = issue_pv(it - 1);
      }
      if (ok) issue_pv(nblk - 1);
      // Teardown: wait for every MMA this thread issued.
      mma_commit(bar_drain);
      drain_wait(bar_drain, 0, p.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warps 0-3
    const int r = threadIdx.x;  // row within the tile == TMEM lane
    const int row_g = row0 + r;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t t_o = tmem + lane_base + L::kColO;
    const float sl2 = p.scale_log2;
    float m_old = -INFINITY;
    float l = 0.f;
    bool alive = true;
    for (int it = 0; it < nblk; ++it) {
      const int b = it & 1;
      if (!warp_wait(&bar_sfull[b], (it >> 1) & 1, abort_flag, p.err, kErrTimeoutSoftmax)) {
        alive = false;
        break;
      }
      tc_fence_after();
      const uint32_t t_s = tmem + lane_base + 128u * b;
      uint32_t sr[kBlockN];
#pragma unroll
      for (int c = 0; c < kBlockN / 32; ++c) tmem_ld32(t_s + c * 32, sr + c * 32);

      const int kv0 = it * kBlockN;
      const bool need_mask = (kv0 + kBlockN > S) || (p.causal && kv0 + kBlockN - 1 > row0);
      if (need_mask) {
        const int last = p.causal ? min(S - 1, row_g) : S - 1;  // last visible key of this row
#pragma unroll
        for (int c = 0; c < kBlockN; ++c)
          if (kv0 + c > last) sr[c] = __float_as_uint(-INFINITY);
      }
      float mx;
      if (sl2 >= 0.f) {
        mx = __uint_as_float(sr[0]);
#pragma unroll
        for (int c = 1; c < kBlockN; ++c) mx = fmaxf(mx, __uint_as_float(sr[c]));
      } else {
        // A negative scale flips the order: the largest scaled score is the smallest raw one.
        mx = INFINITY;
#pragma unroll
        for (int c = 0; c < kBlockN; ++c) {
          const float x = __uint_as_float(sr[c]);
          if (x != -INFINITY) mx = fminf(mx, x);
        }
        if (mx == INFINITY) mx = -INFINITY;
      }
      const float m_blk = (mx == -INFINITY) ? -INFINITY : mx * sl2;
      const float m_new = fmaxf(m_old, m_blk);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = (m_new == m_old) ? 1.f : ex2(m_old - m_use);
      float sum0 = 0.f, sum1 = 0.f;
      uint32_t pk[kBlockN / 2];
#pragma unroll
      for (int c = 0; c < kBlockN / 2; ++c) {
        const float x0 = __uint_as_float(sr[2 * c]);
        const float x1 = __uint_as_float(sr[2 * c + 1]);
        const float p0 = (x0 == -INFINITY) ? 0.f : ex2(fmaf(x0, sl2, -m_use));
        const float p1 = (x1 == -INFINITY) ? 0.f : ex2(fmaf(x1, sl2, -m_use));
        sum0 += p0;
        sum1 += p1;
        pk[c] = pack2<BF16>(p0, p1);
      }
      l = l * alpha + (sum0 + sum1);
      // P (16-bit) overwrites the first 64 columns of this S buffer.
      tmem_st32(t_s, pk);
      tmem_st32(t_s + 32, pk + 32);
      tmem_st_wait();
      if (it > 0 && __any_sync(0xffffffffu, m_new != m_old)) {
        // O holds sum over earlier blocks relative to m_old: wait for the last
        // P V product, then rescale the rows of this warp by alpha.
        if (!warp_wait(&bar_pvdone[(it - 1) & 1], ((it - 1) >> 1) & 1, abort_flag, p.err, kErrTimeoutSoftmax)) {
          alive = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D; c += 16) {
          uint32_t o16[16];
          tmem_ld16(t_o + c, o16);
#pragma unroll
          for (int i = 0; i < 16; ++i) o16[i] = __float_as_uint(__uint_as_float(o16[i]) * alpha);
          tmem_st16(t_o + c, o16);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(&bar_pfull[b]);
      m_old = m_new;
    }
    // ------------------------------------------------------------ epilogue
    if (alive) {
      const int last = nblk - 1;
      if (warp_wait(&bar_pvdone[last & 1], (last >> 1) & 1, abort_flag, p.err, kErrTimeoutSoftmax)) {
        tc_fence_after();
        const float inv_l = 1.f / l;
        const bool row_ok = row_g < S;
        elem_t* orow = reinterpret_cast<elem_t*>(p.o) + (static_cast<size_t>(bh) * S + (row_ok ? row_g : 0)) * D;
#pragma unroll
        for (int c = 0; c < D; c += 16) {
          uint32_t o16[16];
          tmem_ld16(t_o + c, o16);
          uint32_t w[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            w[i] = pack2<BF16>(__uint_as_float(o16[2 * i]) * inv_l, __uint_as_float(o16[2 * i + 1]) * inv_l);
          if (row_ok) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
          }
        }
        if (row_ok) p.lse[static_cast<size_t>(bh) * S + row_g] = (m_old + log2f(l)) * 0.69314718055994530942f;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

namespace {
template <int D, bool BF16>
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                         int BH, cudaStream_t stream) {
  using L = FwdLayout<D>;
  auto kern = fa_fwd_kernel<D, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(BH, p.n_m_tiles);
  kern<<<grid, 192, L::kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_fwd(int D, bool bf16, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, int BH, cudaStream_t stream) {
#define FA_FWD_CASE(DD)                                                  \
  case DD:                                                               \
    return bf16 ? launch_fwd_t<DD, true>(tq, tk, tv, p, BH, stream)      \
                : launch_fwd_t<DD, false>(tq, tk, tv, p, BH, stream);
  switch (D) {
    FA_FWD_CASE(16)
    FA_FWD_CASE(32)
    FA_FWD_CASE(64)
    FA_FWD_CASE(128)
    default:
      return cudaErrorInvalidValue;
  }
#undef FA_FWD_CASE
}

}  // namespace fa
