// Backward kernels: recompute backward of exact attention.
//
// With P = exp(S - L) rebuilt from the forward's logsumexp ("从零训练语言模型
// （第二部分）" §使用 LSE 连接正向和反向传播) and the row vector
// Delta_i = rowsum(dO o O) (CS336 Assignment 2 write-up, "4. Problem
// (flash_backward)", the vector D):
//   dV = P^T dO,   dP = dO V^T,   dS = P o (dP - Delta),
//   dQ = scale * dS K,   dK = scale * dS^T Q          ("第二部分" §反向传播).
//
// Three launches (the two-kernel split of the CS336 write-up, "6.
// FlashAttention-2 Leaderboard", which avoids atomics):
//   1. bwd_preprocess: Delta for every row (memory-bound, one pass over O, dO);
//   2. bwd_main<KV_OUTER = true>:  one CTA per (b*h, 128-key tile), looping
//      over the query tiles that see it; accumulates dV and dK in TMEM;
//   3. bwd_main<KV_OUTER = false>: one CTA per (b*h, 128-query tile), looping
//      over its visible key tiles; accumulates dQ in TMEM.
// Causal: a key tile starts at the diagonal query tile, a query tile stops at
// the diagonal key tile (CS336 write-up, causal tile skipping); the mask is
// applied element-wise only on the diagonal tile and on ragged tails.
//
// bwd_main is written once for both passes.  In each iteration it computes
// two score-shaped products with the CTA's resident tiles A1, A2 as the MMA
// A operands and the streamed tiles B1, B2 as B operands:
//   X = A1 B1^T,  Y = A2 B2^T
//     dK/dV pass: A1 = K, A2 = V, B1 = Q_i, B2 = dO_i -> X = S^T, Y = dP^T
//     dQ pass:    A1 = Q, A2 = dO, B1 = K_j, B2 = V_j -> X = S,   Y = dP
// so TMEM lane = the CTA's own row (key or query) and each softmax thread owns
// a whole row.  The softmax warps turn X, Y into P and dS (16-bit, written
// back into TMEM over X and Y), then the MMA warp accumulates
//     dK/dV pass: dV += P^T dO_i,  dK += dS^T Q_i   (A from TMEM, B = B2, B1 MN-major)
//     dQ pass:    dQ += dS K_j                      (A from TMEM, B = B1 MN-major)
#include "fa_kernel_common.cuh"

namespace fa {
using namespace ptx;

// ------------------------------------------------------------------ preprocess
// Delta_i = sum_d dO_id * O_id in fp32.  D/8 threads share a row, each
// reading 16 bytes of O and of dO; a shuffle tree sums the group.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_preprocess_kernel(const BwdParams p, int64_t rows) {
  constexpr int kTpr = D / 8;           // threads per row
  constexpr int kRowsPerWarp = 32 / kTpr;
  const int lane = threadIdx.x & 31;
  const int sub = lane % kTpr;
  const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  // Whole warps iterate together so the shuffles below always see 32 lanes.
  for (int64_t r0 = warp_id * kRowsPerWarp; r0 < rows; r0 += n_warps * kRowsPerWarp) {
    const int64_t row = r0 + lane / kTpr;
    float acc = 0.f;
    if (row < rows) {
      const uint4 a = reinterpret_cast<const uint4*>(static_cast<const char*>(p.o) + (row * D + sub * 8) * 2)[0];
      const uint4 b = reinterpret_cast<const uint4*>(static_cast<const char*>(p.dout) + (row * D + sub * 8) * 2)[0];
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
      const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float2 fa2, fb2;
        if constexpr (BF16) {
          fa2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&aw[i]));
          fb2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bw[i]));
        } else {
          fa2 = __half22float2(*reinterpret_cast<const __half2*>(&aw[i]));
          fb2 = __half22float2(*reinterpret_cast<const __half2*>(&bw[i]));
        }
        acc = fmaf(fa2.x, fb2.x, acc);
        acc = fmaf(fa2.y, fb2.y, acc);
      }
    }
#pragma unroll
    for (int off = kTpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (row < rows && sub == 0) p.delta[row] = acc;
  }
}

namespace {

template <int D, bool KV_OUTER>
struct BwdLayout : TileGeom<D> {
  using G = TileGeom<D>;
  static constexpr int kStages = 2;
  static constexpr int kOffA1 = 0;
  static constexpr int kOffA2 = kOffA1 + G::kTileBytes;
  static constexpr int kOffB1 = kOffA2 + G::kTileBytes;                  // [kStages] tiles
  static constexpr int kOffB2 = kOffB1 + kStages * G::kTileBytes;        // [kStages] tiles
  static constexpr int kOffRowVec = kOffB2 + kStages * G::kTileBytes;    // [2][2][128] fp32: L2, Delta per column
  static constexpr int kOffBar = kOffRowVec + 2 * 2 * 128 * 4;
  // a_full, b_full[S], empty[S], xy_full, p_full, acc_done, drain
  static constexpr int kNumBars = 1 + 2 * kStages + 4;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemUsed = kOffMisc + 16;
  static constexpr int kSmemBytes = (kSmemUsed + 1024) > 116 * 1024 ? (kSmemUsed + 1024) : 116 * 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColX = 0;     // S or S^T; P^T overwrites its first 64 columns
  static constexpr uint32_t kColY = 128;   // dP or dP^T; dS (dS^T) overwrites its first 64 columns
  static constexpr uint32_t kColAcc1 = 256;                 // dV (dK/dV pass) or dQ
  static constexpr uint32_t kColAcc2 = 384;                 // dK (dK/dV pass)
};

}  // namespace

template <int D, bool BF16, bool KV_OUTER>
__global__ void __launch_bounds__(192, 1)
    fa_bwd_main_kernel(const __grid_constant__ CUtensorMap tm_a1, const __grid_constant__ CUtensorMap tm_a2,
                       const __grid_constant__ CUtensorMap tm_b1, const __grid_constant__ CUtensorMap tm_b2,
                       const BwdParams p) {
  using L = BwdLayout<D, KV_OUTER>;
  using elem_t = typename std::conditional<BF16, __nv_bfloat16, __half>::type;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* bar_afull = bars;
  uint64_t* bar_bfull = bars + 1;
  uint64_t* bar_empty = bar_bfull + L::kStages;
  uint64_t* bar_xyfull = bar_empty + L::kStages;
  uint64_t* bar_pfull = bar_xyfull + 1;
  uint64_t* bar_accdone = bar_pfull + 1;
  uint64_t* bar_drain = bar_accdone + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);
  float* rowvec = reinterpret_cast<float*>(smem + L::kOffRowVec);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int S = p.S;
  const int nt = p.n_tiles;
  // Own tile; heavy tiles first under the causal mask (key tile 0 and query
  // tile nt-1 see the most partners).
  const int own = KV_OUTER ? static_cast<int>(blockIdx.y)
                           : (p.causal ? nt - 1 - static_cast<int>(blockIdx.y) : static_cast<int>(blockIdx.y));
  const int first = (KV_OUTER && p.causal) ? own : 0;
  const int last_excl = (!KV_OUTER && p.causal) ? own + 1 : nt;
  const int niter = last_excl - first;
  const int own0 = own * 128;

  if (threadIdx.x == 0) {
    mbar_init(bar_afull, 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(&bar_bfull[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    mbar_init(bar_xyfull, 1);
    mbar_init(bar_pfull, 128);
    mbar_init(bar_accdone, 1);
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
  const uint32_t sA1 = smem_u32(smem + L::kOffA1);
  const uint32_t sA2 = smem_u32(smem + L::kOffA2);
  const uint32_t sB1 = smem_u32(smem + L::kOffB1);
  const uint32_t sB2 = smem_u32(smem + L::kOffB2);

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_a1);
      prefetch_tmap(&tm_a2);
      prefetch_tmap(&tm_b1);
      prefetch_tmap(&tm_b2);
      mbar_arrive_expect_tx(bar_afull, 2 * L::kTileBytes);
#pragma unroll
      for (int ch = 0; ch < L::kChunks; ++ch) {
        tma_load_3d(smem + L::kOffA1 + ch * L::kChunkBytes, &tm_a1, bar_afull, ch * (L::kRowBytes / 2), own0, bh);
        tma_load_3d(smem + L::kOffA2 + ch * L::kChunkBytes, &tm_a2, bar_afull, ch * (L::kRowBytes / 2), own0, bh);
      }
      int it = 0;
      for (; it < niter; ++it) {
        const int st = it % L::kStages;
        const int use = it / L::kStages;
        if (use > 0 && !mbar_wait(&bar_empty[st], (use - 1) & 1, abort_flag, p.err, kErrTimeoutLoad)) break;
        const int r0 = (first + it) * 128;
        mbar_arrive_expect_tx(&bar_bfull[st], 2 * L::kTileBytes);
#pragma unroll
        for (int ch = 0; ch < L::kChunks; ++ch) {
          tma_load_3d(smem + L::kOffB1 + st * L::kTileBytes + ch * L::kChunkBytes, &tm_b1, &bar_bfull[st],
                      ch * (L::kRowBytes / 2), r0, bh);
          tma_load_3d(smem + L::kOffB2 + st * L::kTileBytes + ch * L::kChunkBytes, &tm_b2, &bar_bfull[st],
                      ch * (L::kRowBytes / 2), r0, bh);
        }
      }
      drain_wait(bar_afull, 0, p.err);
      for (int x = (it > L::kStages ? it - L::kStages : 0); x < it; ++x)
        drain_wait(&bar_bfull[x % L::kStages], (x / L::kStages) & 1, p.err);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_xy = make_idesc_f16(BF16, 128, 128, false, false);
      constexpr uint32_t idesc_acc = make_idesc_f16(BF16, 128, D, false, true);
      bool ok = mbar_wait(bar_afull, 0, abort_flag, p.err, kErrTimeoutMma);
      for (int it = 0; ok && it < niter; ++it) {
        const int st = it % L::kStages;
        ok = mbar_wait(&bar_bfull[st], (it / L::kStages) & 1, abort_flag, p.err, kErrTimeoutMma);
        // X and Y are overwritten below: the previous iteration's accumulation
        // (which reads P and dS from them) must be complete.
        if (ok && it > 0) ok = mbar_wait(bar_accdone, (it - 1) & 1, abort_flag, p.err, kErrTimeoutMma);
        if (!ok) break;
        tc_fence_after();
        const uint32_t b1 = sB1 + st * L::kTileBytes;
        const uint32_t b2 = sB2 + st * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + L::kColX, kmajor_desc<D>(sA1, kk), kmajor_desc<D>(b1, kk), idesc_xy, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss(tmem + L::kColY, kmajor_desc<D>(sA2, kk), kmajor_desc<D>(b2, kk), idesc_xy, kk > 0 ? 1u : 0u);
        mma_commit(bar_xyfull);
        ok = mbar_wait(bar_pfull, it & 1, abort_flag, p.err, kErrTimeoutMma);
        if (!ok) break;
        tc_fence_after();
        if constexpr (KV_OUTER) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // dV += P^T dO_i
            mma_ts(tmem + L::kColAcc1, tmem + L::kColX + kk * 8, mnmajor_desc<D>(b2, kk), idesc_acc,
                   (it > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // dK += dS^T Q_i
            mma_ts(tmem + L::kColAcc2, tmem + L::kColY + kk * 8, mnmajor_desc<D>(b1, kk), idesc_acc,
                   (it > 0 || kk > 0) ? 1u : 0u);
        } else {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // dQ += dS K_j
            mma_ts(tmem + L::kColAcc1, tmem + L::kColY + kk * 8, mnmajor_desc<D>(b1, kk), idesc_acc,
                   (it > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&bar_empty[st]);
        mma_commit(bar_accdone);
      }
      mma_commit(bar_drain);
      drain_wait(bar_drain, 0, p.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax-gradient warps 0-3
    const int r = threadIdx.x;
    const int my = own0 + r;  // key index (dK/dV pass) or query index (dQ pass)
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tX = tmem + lane_base + L::kColX;
    const uint32_t tY = tmem + lane_base + L::kColY;
    const float sl2 = p.scale_log2;
    constexpr float kLog2e = 1.4426950408889634f;
    const int64_t rowbase = static_cast<int64_t>(bh) * S;
    // dQ pass: this thread's query row owns its L2 = L * log2 e and Delta.
    float my_l2 = INFINITY, my_delta = 0.f;
    if (!KV_OUTER && my < S) {
      my_l2 = p.lse[rowbase + my] * kLog2e;
      my_delta = p.delta[rowbase + my];
    }
    bool alive = true;
    for (int it = 0; it < niter; ++it) {
      const int other0 = (first + it) * 128;
      float* l2v = rowvec + (it & 1) * 256;
      float* dlv = l2v + 128;
      if constexpr (KV_OUTER) {
        // Per-column (query) L2 and Delta for this query tile; queries past S
        // get L2 = +inf, so their probabilities are exactly 0.
        const int q = other0 + r;
        l2v[r] = q < S ? p.lse[rowbase + q] * kLog2e : INFINITY;
        dlv[r] = q < S ? p.delta[rowbase + q] : 0.f;
      }
      // One barrier over the 128 threads publishes the column vectors and
      // makes the outcome of the wait uniform, so no thread is ever left
      // waiting at a barrier that the others have abandoned.
      const bool got = mbar_wait(bar_xyfull, it & 1, abort_flag, p.err, kErrTimeoutSoftmax);
      if (!named_sync_and(1, 128, got)) {
        alive = false;
        break;
      }
      tc_fence_after();
      // Masked tiles: the diagonal under the causal mask, and a tile of
      // partner rows that runs past S (keys past S in the dQ pass).
      const bool diag = p.causal && (other0 == own0);
      const bool tail = !KV_OUTER && (other0 + 128 > S);
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
        uint32_t xs[32], ys[32];
        tmem_ld32(tX + c0, xs);
        tmem_ld32(tY + c0, ys);
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float pr[2], ds[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int col = c0 + c + u;
            const float l2 = KV_OUTER ? l2v[col] : my_l2;
            const float dl = KV_OUTER ? dlv[col] : my_delta;
            float pv = ex2(fmaf(__uint_as_float(xs[c + u]), sl2, -l2));
            if (diag || tail) {
              const int key = KV_OUTER ? my : other0 + col;
              const int qry = KV_OUTER ? other0 + col : my;
              if ((p.causal && key > qry) || key >= S) pv = 0.f;
            }
            pr[u] = pv;
            ds[u] = pv * (__uint_as_float(ys[c + u]) - dl);
          }
          pk[c / 2] = pack2<BF16>(pr[0], pr[1]);
          dk[c / 2] = pack2<BF16>(ds[0], ds[1]);
        }
        // 16-bit P (dK/dV pass only) and dS go over columns already consumed.
        if constexpr (KV_OUTER) tmem_st16(tX + c0 / 2, pk);
        tmem_st16(tY + c0 / 2, dk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(bar_pfull);
    }
    // ------------------------------------------------------------ epilogue
    const bool done = alive && mbar_wait(bar_accdone, (niter - 1) & 1, abort_flag, p.err, kErrTimeoutSoftmax);
    if (__all_sync(0xffffffffu, done)) {
      tc_fence_after();
      const bool row_ok = my < S;
      const size_t off = (static_cast<size_t>(rowbase) + (row_ok ? my : 0)) * D;
      if constexpr (KV_OUTER) {
        elem_t* dv_row = reinterpret_cast<elem_t*>(p.dv) + off;
        elem_t* dk_row = reinterpret_cast<elem_t*>(p.dk) + off;
#pragma unroll
        for (int c = 0; c < D; c += 16) {
          uint32_t v16[16];
          tmem_ld16(tmem + lane_base + L::kColAcc1 + c, v16);
          if (row_ok) store_row16<BF16>(dv_row + c, v16, 1.f);
          tmem_ld16(tmem + lane_base + L::kColAcc2 + c, v16);
          if (row_ok) store_row16<BF16>(dk_row + c, v16, p.scale);
        }
      } else {
        elem_t* dq_row = reinterpret_cast<elem_t*>(p.dq) + off;
#pragma unroll
        for (int c = 0; c < D; c += 16) {
          uint32_t v16[16];
          tmem_ld16(tmem + lane_base + L::kColAcc1 + c, v16);
          if (row_ok) store_row16<BF16>(dq_row + c, v16, p.scale);
        }
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
cudaError_t launch_pre_t(const BwdParams& p, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(p.BH) * p.S;
  const int64_t threads = rows * (D / 8);
  const int64_t blocks = (threads + 255) / 256;
  const int grid = static_cast<int>(blocks < 152 * 16 ? blocks : 152 * 16);
  fa_bwd_preprocess_kernel<D, BF16><<<grid, 256, 0, stream>>>(p, rows);
  return cudaGetLastError();
}

template <int D, bool BF16, bool KV_OUTER>
cudaError_t launch_main_t(const CUtensorMap& a1, const CUtensorMap& a2, const CUtensorMap& b1,
                          const CUtensorMap& b2, const BwdParams& p, cudaStream_t stream) {
  using L = BwdLayout<D, KV_OUTER>;
  auto kern = fa_bwd_main_kernel<D, BF16, KV_OUTER>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(p.BH, p.n_tiles);
  kern<<<grid, 192, L::kSmemBytes, stream>>>(a1, a2, b1, b2, p);
  return cudaGetLastError();
}

}  // namespace

#define FA_BWD_DISPATCH(CALL)                              \
  switch (D) {                                             \
    case 16: return bf16 ? CALL(16, true) : CALL(16, false);   \
    case 32: return bf16 ? CALL(32, true) : CALL(32, false);   \
    case 64: return bf16 ? CALL(64, true) : CALL(64, false);   \
    case 128: return bf16 ? CALL(128, true) : CALL(128, false); \
    default: return cudaErrorInvalidValue;                 \
  }

cudaError_t launch_bwd_preprocess(int D, bool bf16, const BwdParams& p, cudaStream_t stream) {
#define FA_PRE(DD, BB) launch_pre_t<DD, BB>(p, stream)
  FA_BWD_DISPATCH(FA_PRE)
#undef FA_PRE
}

cudaError_t launch_bwd_dkdv(int D, bool bf16, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const BwdParams& p, cudaStream_t stream) {
#define FA_DKDV(DD, BB) launch_main_t<DD, BB, true>(tk, tv, tq, tdo, p, stream)
  FA_BWD_DISPATCH(FA_DKDV)
#undef FA_DKDV
}

cudaError_t launch_bwd_dq(int D, bool bf16, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const BwdParams& p, cudaStream_t stream) {
#define FA_DQ(DD, BB) launch_main_t<DD, BB, false>(tq, tdo, tk, tv, p, stream)
  FA_BWD_DISPATCH(FA_DQ)
#undef FA_DQ
}

#undef FA_BWD_DISPATCH

}  // namespace fa
