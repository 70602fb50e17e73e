// Forward kernel: exact attention with an online softmax, FlashAttention-2
// loop order (query block outer, key/value block inner), on tcgen05 tensor
// cores with accumulators in tensor memory (TMEM).
//
// One CTA per (batch*head, 256 query rows) = two 128-row query tiles that
// share every K/V block the CTA loads.  Warp roles (384 threads):
//   warps 0-3  softmax warpgroup of tile 0, warps 4-7 that of tile 1; thread
//              t of a warpgroup owns query row t of its tile = TMEM lane t, so
//              row max and row sum need no cross-thread reduction (the split-Q
//              partition of "Inside FlashAttention" §4.3);
//   warp 8     TMA producer: both Q tiles once, then K and V blocks through a
//              ring of shared-memory stages (warps 10-11 idle; warps 8-11 give
//              their registers to the softmax warpgroups with setmaxnreg);
//   warp 9     MMA issuer.  Per key block j it issues, in this order,
//              O0 += P0(j-1) V(j-1), S0 = Q0 K(j)^T, O1 += P1(j-1) V(j-1),
//              S1 = Q1 K(j)^T, so while one warpgroup runs the softmax of its
//              tile the tensor core works on the other tile (the warp
//              specialisation and matmul/softmax overlap of "Inside
//              FlashAttention" §5.1-5.2).
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+D), O1 after it.
// P (16-bit) is written over the first 64 columns of its tile's S and read
// by the P V MMA straight from TMEM.  The tensor core runs one CTA's MMAs in
// issue order, so S(j+1) is written only after P(j) V(j) has read P(j).
//
// Per key block j, per row, in the base-2 domain (c = scale * log2 e):
//   m_blk = c * rowmax(S_j)                        ("T5 讲解" §④; "fa-triton" Step 2)
//   if m_blk > m + tau: alpha = exp2(m - m_blk), m = m_blk, l *= alpha, O *= alpha
//   P~ = exp2(c * S_j - m),  l += rowsum(P~),  O += P~ V_j    ("fa-triton" Steps 3-4)
// Keeping a stale m while the block maximum exceeds it by at most tau = 8
// is exact in real arithmetic (P~ <= 2^8 stays well inside the 16-bit range)
// and rescales O only when the maximum really moves ("Inside FlashAttention"
// §4.1: fewer non-matmul operations).  Epilogue: O / l and L = (m + log2 l) ln 2.
//
// Causal: tile t of query rows visits key blocks up to its diagonal block
// ("T5 讲解" §⑤); masking is element-wise only on the diagonal block and on a
// ragged last key block ("fa-triton" §Causal Mask 的处理：off-band 与 on-band).
#include "fa_kernel_common.cuh"

namespace fa {
using namespace ptx;

namespace {

constexpr int kFwdThreads = 384;
// Register split (per thread): the launch gives every thread kLaunchRegs; the
// producer/MMA warpgroup drops to kRegsLow and both softmax warpgroups rise
// to kRegsHigh.  2 * 128 * kRegsHigh + 128 * kRegsLow == 384 * kLaunchRegs.
constexpr int kLaunchRegs = 168;
constexpr uint32_t kRegsHigh = 224;
constexpr uint32_t kRegsLow = 56;
static_assert(2 * 128 * kRegsHigh + 128 * kRegsLow == kFwdThreads * kLaunchRegs, "register split");
constexpr float kTau = 8.0f;  // stale-max threshold (log2 units)

template <int D>
struct FwdLayout : TileGeom<D> {
  using G = TileGeom<D>;
  static constexpr int kStages = D <= 64 ? 3 : 2;
  static constexpr int kOffQ = 0;  // two query tiles
  static constexpr int kOffK = kOffQ + 2 * G::kTileBytes;
  static constexpr int kOffV = kOffK + kStages * G::kTileBytes;
  static constexpr int kOffBar = kOffV + kStages * G::kTileBytes;
  // q, kfull[S], vfull[S], empty[S], sfull[2], pfull[2], ofinal[2], drain
  static constexpr int kNumBars = 1 + 3 * kStages + 6 + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemUsed = kOffMisc + 16;
  // Tensor memory is allocated whole (512 columns), so at most one CTA may
  // live on an SM: the request is padded above half of the SM's shared memory.
  static constexpr int kSmemBytes = (kSmemUsed + 1024) > 116 * 1024 ? (kSmemUsed + 1024) : 116 * 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 256;  // O0 at 256, O1 at 256 + D
};

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

}  // namespace

template <int D, bool BF16>
__global__ void __launch_bounds__(kFwdThreads, 1)
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
  uint64_t* bar_sfull = bar_empty + L::kStages;  // [2] per tile
  uint64_t* bar_pfull = bar_sfull + 2;           // [2]
  uint64_t* bar_ofinal = bar_pfull + 2;          // [2]
  uint64_t* bar_drain = bar_ofinal + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int S = p.S;
  const int cta = p.causal ? (p.n_m_tiles - 1 - static_cast<int>(blockIdx.y)) : static_cast<int>(blockIdx.y);
  const int row0 = cta * 2 * kBlockM;
  const int n_kv = (S + kBlockN - 1) / kBlockN;
  // Key blocks visited by each tile (tile 1 sees at most one more under the mask).
  const int nb0 = p.causal ? min(n_kv, (row0 + kBlockM + kBlockN - 1) / kBlockN) : n_kv;
  const int nb1 = p.causal ? min(n_kv, (row0 + 2 * kBlockM + kBlockN - 1) / kBlockN) : n_kv;

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(&bar_kfull[s], 1);
      mbar_init(&bar_vfull[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bar_sfull[t], 1);
      mbar_init(&bar_pfull[t], 128);
      mbar_init(&bar_ofinal[t], 1);
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
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

  if (warp >= 8) {
    regs_decrease<kRegsLow>();
    if (warp == 8) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        mbar_arrive_expect_tx(bar_q, 2 * L::kTileBytes);
  #pragma unroll
        for (int t = 0; t < 2; ++t)
  #pragma unroll
          for (int ch = 0; ch < L::kChunks; ++ch)
            tma_load_3d(smem + L::kOffQ + t * L::kTileBytes + ch * L::kChunkBytes, &tm_q, bar_q,
                        ch * (L::kRowBytes / 2), row0 + t * kBlockM, bh);
        int it = 0;
        for (; it < nb1; ++it) {
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
    } else if (warp == 9) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        constexpr uint32_t idesc_qk = make_idesc_f16(BF16, 128, kBlockN, false, false);
        constexpr uint32_t idesc_pv = make_idesc_f16(BF16, 128, D, false, true);
        auto qk = [&](int t, int j) {
          const uint32_t k_addr = sK + (j % L::kStages) * L::kTileBytes;
          const uint32_t q_addr = sQ + t * L::kTileBytes;
  #pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(tmem + 128u * t, kmajor_desc<D>(q_addr, kk), kmajor_desc<D>(k_addr, kk), idesc_qk,
                   kk > 0 ? 1u : 0u);
          mma_commit(&bar_sfull[t]);
        };
        auto pv = [&](int t, int j) -> bool {
          const int st = j % L::kStages;
          if (!mbar_wait(&bar_pfull[t], j & 1, abort_flag, p.err, kErrTimeoutMma)) return false;
          if (!mbar_wait(&bar_vfull[st], (j / L::kStages) & 1, abort_flag, p.err, kErrTimeoutMma)) return false;
          tc_fence_after();
          const uint32_t v_addr = sV + st * L::kTileBytes;
  #pragma unroll
          for (int kk = 0; kk < kBlockN / 16; ++kk)
            mma_ts(tmem + L::kColO + D * t, tmem + 128u * t + kk * 8, mnmajor_desc<D>(v_addr, kk), idesc_pv,
                   (j > 0 || kk > 0) ? 1u : 0u);
          return true;
        };
        bool ok = mbar_wait(bar_q, 0, abort_flag, p.err, kErrTimeoutMma);
        for (int j = 0; ok && j < nb1; ++j) {
          const int st = j % L::kStages;
          ok = mbar_wait(&bar_kfull[st], (j / L::kStages) & 1, abort_flag, p.err, kErrTimeoutMma);
          if (!ok) break;
          tc_fence_after();
          if (j >= 1 && j - 1 < nb0) {
            if (!(ok = pv(0, j - 1))) break;
            if (j - 1 == nb0 - 1) mma_commit(&bar_ofinal[0]);
          }
          if (j < nb0) qk(0, j);
          if (j >= 1) {
            if (!(ok = pv(1, j - 1))) break;
            mma_commit(&bar_empty[(j - 1) % L::kStages]);
          }
          qk(1, j);
        }
        if (ok && nb0 == nb1) {
          ok = pv(0, nb0 - 1);
          if (ok) mma_commit(&bar_ofinal[0]);
        }
        if (ok && pv(1, nb1 - 1)) mma_commit(&bar_ofinal[1]);
        // Teardown: wait for every MMA this thread issued.
        mma_commit(bar_drain);
        drain_wait(bar_drain, 0, p.err);
      }
      __syncwarp();
    }
  } else {
    regs_increase<kRegsHigh>();
    // ------------------------------------------------------------ softmax warpgroups
    const int t = warp >> 2;            // tile
    const int r = threadIdx.x & 127;    // row within the tile == TMEM lane
    const int tile_row0 = row0 + t * kBlockM;
    const int row_g = tile_row0 + r;
    const int nb = t == 0 ? nb0 : nb1;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lane_base + 128u * t;
    const uint32_t t_o = tmem + lane_base + L::kColO + D * t;
    const float sl2 = p.scale_log2;
    const float2 c2 = make_float2(sl2, sl2);
    // last visible key of this row
    const int last = p.causal ? min(S - 1, row_g) : S - 1;
    float m = -INFINITY;  // running (possibly stale) maximum, base-2 scaled
    float l = 0.f;
    bool alive = true;
    for (int j = 0; j < nb; ++j) {
      if (!warp_wait(&bar_sfull[t], j & 1, abort_flag, p.err, kErrTimeoutSoftmax)) {
        alive = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[kBlockN];
      tmem_ld128(t_s, sr);
      const int kv0 = j * kBlockN;
      // Masked blocks: the diagonal block under the causal mask, and a
      // ragged last key block.
      const bool masked = (kv0 + kBlockN > S) || (p.causal && kv0 + kBlockN - 1 > tile_row0);
      float mx;
      if (!masked) {
        float a = __uint_as_float(sr[0]), b = __uint_as_float(sr[1]);
        if (sl2 >= 0.f) {
#pragma unroll
          for (int c = 2; c < kBlockN - 2; c += 4) {
            a = max3(a, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
            b = max3(b, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
          }
          mx = max3(a, b, fmaxf(__uint_as_float(sr[kBlockN - 2]), __uint_as_float(sr[kBlockN - 1])));
        } else {  // a negative scale turns the largest scaled score into the smallest raw one
#pragma unroll
          for (int c = 2; c < kBlockN - 2; c += 4) {
            a = min3(a, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
            b = min3(b, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
          }
          mx = min3(a, b, fminf(__uint_as_float(sr[kBlockN - 2]), __uint_as_float(sr[kBlockN - 1])));
        }
      } else {
        mx = sl2 >= 0.f ? -INFINITY : INFINITY;
#pragma unroll
        for (int c = 0; c < kBlockN; ++c) {
          const float x = __uint_as_float(sr[c]);
          if (kv0 + c <= last) mx = sl2 >= 0.f ? fmaxf(mx, x) : fminf(mx, x);
        }
      }
      // A block with no visible key for this row (only rows past S) contributes nothing.
      const float m_blk = (kv0 > last) ? -INFINITY : mx * sl2;
      float alpha = 1.f;
      bool upd = false;
      if (j == 0) {
        m = m_blk;
      } else if (m_blk > m + kTau) {
        alpha = ex2(m - m_blk);
        m = m_blk;
        upd = true;
      }
      if (__any_sync(0xffffffffu, upd)) {
        // O holds the blocks before j, relative to the old m.  The commit
        // that signalled S(j) also covers the earlier P V MMA, so O is final.
        l *= alpha;
#pragma unroll
        for (int c = 0; c < D; c += 16) {
          uint32_t o16[16];
          tmem_ld16(t_o + c, o16);
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            const float2 v = __fmul2_rn(make_float2(__uint_as_float(o16[i]), __uint_as_float(o16[i + 1])),
                                        make_float2(alpha, alpha));
            o16[i] = __float_as_uint(v.x);
            o16[i + 1] = __float_as_uint(v.y);
          }
          tmem_st16(t_o + c, o16);
        }
      }
      const float m_use = (m == -INFINITY) ? 0.f : m;
      const float2 negm = make_float2(-m_use, -m_use);
      float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
      // P (16-bit) overwrites the first 64 columns of this tile's S, 16 columns
      // (32 scores) at a time, so only the S row itself stays live in registers.
      if (!masked) {
#pragma unroll
        for (int c0 = 0; c0 < kBlockN; c0 += 32) {
          uint32_t pk[16];
#pragma unroll
          for (int c = c0; c < c0 + 32; c += 4) {
            const float2 y0 =
                __ffma2_rn(make_float2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), c2, negm);
            const float2 y1 =
                __ffma2_rn(make_float2(__uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3])), c2, negm);
            const float2 e0 = make_float2(ex2(y0.x), ex2(y0.y));
            const float2 e1 = make_float2(ex2(y1.x), ex2(y1.y));
            acc0 = __fadd2_rn(acc0, e0);
            acc1 = __fadd2_rn(acc1, e1);
            pk[(c - c0) / 2] = pack2<BF16>(e0.x, e0.y);
            pk[(c - c0) / 2 + 1] = pack2<BF16>(e1.x, e1.y);
          }
          tmem_st16(t_s + c0 / 2, pk);
        }
      } else {
#pragma unroll
        for (int c0 = 0; c0 < kBlockN; c0 += 32) {
          uint32_t pk[16];
#pragma unroll
          for (int c = c0; c < c0 + 32; c += 2) {
            const float2 y =
                __ffma2_rn(make_float2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), c2, negm);
            const float e0 = (kv0 + c <= last) ? ex2(y.x) : 0.f;
            const float e1 = (kv0 + c + 1 <= last) ? ex2(y.y) : 0.f;
            acc0 = __fadd2_rn(acc0, make_float2(e0, e1));
            pk[(c - c0) / 2] = pack2<BF16>(e0, e1);
          }
          tmem_st16(t_s + c0 / 2, pk);
        }
      }
      const float2 acc = __fadd2_rn(acc0, acc1);
      l += acc.x + acc.y;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bar_pfull[t]);
    }
    // ------------------------------------------------------------ epilogue
    if (alive && warp_wait(&bar_ofinal[t], 0, abort_flag, p.err, kErrTimeoutSoftmax)) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      const bool row_ok = row_g < S;
      elem_t* orow = reinterpret_cast<elem_t*>(p.o) + (static_cast<size_t>(bh) * S + (row_ok ? row_g : 0)) * D;
#pragma unroll
      for (int c = 0; c < D; c += 16) {
        uint32_t o16[16];
        tmem_ld16(t_o + c, o16);
        if (row_ok) store_row16<BF16>(orow + c, o16, inv_l);
      }
      if (row_ok) p.lse[static_cast<size_t>(bh) * S + row_g] = (m + log2f(l)) * 0.69314718055994530942f;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
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
  // The register split above assumes the launch gives exactly kLaunchRegs per
  // thread; with fewer, the softmax warpgroups' increase could never be met.
  cudaFuncAttributes attr;
  e = cudaFuncGetAttributes(&attr, kern);
  if (e != cudaSuccess) return e;
  if (attr.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
  dim3 grid(BH, p.n_m_tiles);
  kern<<<grid, kFwdThreads, L::kSmemBytes, stream>>>(tq, tk, tv, p);
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
