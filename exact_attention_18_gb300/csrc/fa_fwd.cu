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
//              ring of shared-memory stages (warp 11 idle; warps 8-11 give
//              their registers to the softmax warpgroups with setmaxnreg);
//   warps 9-10 MMA issuers, one per tile.
// The two tiles' softmax work overlaps the tensor core's work on the other
// tile (the warp specialisation and matmul/softmax overlap of "Inside
// FlashAttention" §5.1-5.2).
//
// TMEM (512 columns) for D <= 64: S0 [0,128), S1 [128,256), P0 [256,320),
// P1 [320,384), O0 [384,384+D), O1 after it.  P (16-bit) has its own columns,
// so a warpgroup releases S_t(j) as soon as it has loaded it into registers
// and the MMA warp computes S_t(j+1) while the softmax of block j still runs.
// Per key block j the MMA warp issues S0 = Q0 K(j)^T, S1 = Q1 K(j)^T, then
// O0 += P0(j-1) V(j-1), O1 += P1(j-1) V(j-1).
// For D = 128 (O0, O1 take 256 columns) P is written over the first 64
// columns of its S and the order is O0 += P0 V, S0 = Q0 K^T, O1 += P1 V,
// S1 = Q1 K^T; the tensor core runs one CTA's MMAs in issue order, so S(j+1)
// is written only after P(j) V(j) has read P(j).
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
#include "fa_softmax.cuh"

namespace fa {
using namespace ptx;

namespace {

constexpr int kFwdThreads = 384;
// Register split (per thread): the launch gives every thread kLaunchRegs; the
// producer/MMA warpgroup drops to kRegsLow and both softmax warpgroups rise
// to kRegsHigh; the shares may not exceed the launch total 384 * kLaunchRegs.
constexpr int kLaunchRegs = 168;
constexpr uint32_t kRegsHigh = 224;
constexpr uint32_t kRegsLow = 56;
static_assert(2 * 128 * kRegsHigh + 128 * kRegsLow <= kFwdThreads * kLaunchRegs, "register split");
// A block's P~ = exp2(c s - m) is accepted with a stale maximum m while the
// block's sum stays <= 2^8 (so every P~ <= 2^8, far inside the 16-bit range).
constexpr float kSumLimit = 256.0f;
// The two tiles' softmax warps of one SM sub-partition alternate at the
// exponentials of each key block.
constexpr bool kTurns = true;

template <int D>
struct FwdLayout : TileGeom<D> {
  using G = TileGeom<D>;
  static constexpr bool kSepP = D <= 64;  // P in its own TMEM columns
  // K and V blocks travel through separate rings: a K stage is released once
  // both tiles' score products on it are done, a V stage only after both
  // tiles' P V, about half a block later.  With one ring for both, a stage
  // came free so late that the next K block's copy had a few hundred cycles
  // to land; a third K stage adds a whole block of lead.
  static constexpr int kStagesK = 3;
  static constexpr int kStagesV = D <= 64 ? 3 : 2;
  static constexpr int kOffQ = 0;  // two query tiles
  static constexpr int kOffK = kOffQ + 2 * G::kTileBytes;
  static constexpr int kOffV = kOffK + kStagesK * G::kTileBytes;
  static constexpr int kOffBar = kOffV + kStagesV * G::kTileBytes;
  // q, kfull[SK], kempty[SK], vfull[SV], vempty[SV], sfull[2], sfree[2], pfull[2], pvdone[2], ofinal[2],
  // drain[2], turn[8]
  static constexpr int kNumBars = 1 + 2 * kStagesK + 2 * kStagesV + 10 + 2 + 8;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemUsed = kOffMisc + 16;
  // Tensor memory is allocated whole (512 columns), so at most one CTA may
  // live on an SM: the request is padded above half of the SM's shared memory.
  static constexpr int kSmemBytes = (kSmemUsed + 1024) > 116 * 1024 ? (kSmemUsed + 1024) : 116 * 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0;                   // S_t at 128 t
  static constexpr uint32_t kColP = kSepP ? 256 : 0;     // P_t at kColP + (kSepP ? 64 : 128) t
  static constexpr uint32_t kStrideP = kSepP ? 64 : 128;
  static constexpr uint32_t kColO = kSepP ? 384 : 256;   // O_t at kColO + D t
  static_assert(kColO + 2 * D <= kTmemCols, "TMEM layout");
};

// P~ = exp2(c2 * s - m) for the block's 128 scores, packed as 16-bit pairs
// into pk; with `masked`, columns past lim (and, with LO, before lo) are
// exactly 0.  Returns the fp32 sum of the unrounded P~ (the block's share of
// the running sum l).
template <bool BF16, bool LO>
__device__ __forceinline__ float exp_block(const uint32_t* sr, float2 c2, float m, bool masked, int lo, int lim,
                                           uint32_t* pk) {
  const float m_use = (m == -INFINITY) ? 0.f : m;  // rows with no visible key so far
  const float2 negm = make_float2(-m_use, -m_use);
  float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  if (masked) {
#pragma unroll
    for (int k0 = 0; k0 < kBlockN; k0 += 16) exp16<BF16, true, LO>(sr, k0, c2, negm, lo, lim, acc, pk + k0 / 2);
  } else {
#pragma unroll
    for (int k0 = 0; k0 < kBlockN; k0 += 16) exp16<BF16, false>(sr, k0, c2, negm, lo, lim, acc, pk + k0 / 2);
  }
  const float2 a = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
  return a.x + a.y;
}

}  // namespace

// tm_q: 128-row boxes (a CTA's own query tiles); tm_k, tm_v: 64-row boxes
// (each K/V block arrives as two half-block copies).  GENERAL: packed
// batches and windows, as in the four-tile kernel.
template <int D, bool BF16, bool GENERAL>
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
  uint64_t* bar_kempty = bar_kfull + L::kStagesK;
  uint64_t* bar_vfull = bar_kempty + L::kStagesK;
  uint64_t* bar_vempty = bar_vfull + L::kStagesV;
  uint64_t* bar_sfull = bar_vempty + L::kStagesV;  // [2] per tile: S_t(j) computed
  uint64_t* bar_sfree = bar_sfull + 2;           // [2] S_t(j) loaded by its warpgroup (separate-P layout)
  uint64_t* bar_pfull = bar_sfree + 2;           // [2] P_t(j) stored, O_t rescaled
  uint64_t* bar_pvdone = bar_pfull + 2;          // [2] O_t += P_t(j) V(j) done (separate-P layout)
  uint64_t* bar_ofinal = bar_pvdone + 2;         // [2] last P V of tile t done
  uint64_t* bar_drain = bar_ofinal + 2;          // [2] one per MMA warp
  uint64_t* bar_turn = bar_drain + 2;            // [2][4] tile t's warps q may start their exponentials
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);

  const int warp = warp_index();
  const int lane = threadIdx.x & 31;
  int cx, cy;
  cta_coords(!p.causal, &cx, &cy);
  const int bh = cx;
  // General instantiation: the sample of a packed batch (the layouts of
  // FwdParams); q_head / kvh are then heads within a token.
  int S_ = p.S, kvh_ = bh / p.group, q_head = bh, tok0 = 0;
  bool packed = false;
  if constexpr (GENERAL) {
    packed = p.cu_seqlens != nullptr;
    if (packed) {
      const int b = bh / p.heads;
      q_head = bh - b * p.heads;
      kvh_ = q_head / p.group;
      if (!packed_sample(p.cu_seqlens, b, p.S, p.total, p.err, &tok0, &S_)) return;
    }
  }
  const int kvh = kvh_;  // K/V head shared by this query head's group
  const int S = S_;
  // Under the causal mask the heaviest CTAs are launched first.
  const int cta = p.causal ? p.n_m_tiles - 1 - cy : cy;
  const int row0 = cta * 2 * kBlockM;
  if constexpr (GENERAL) {
    if (row0 >= S) return;  // packed batch: this CTA lies past its sample
  }
  const int n_kv = (S + kBlockN - 1) / kBlockN;
  // Window (general instantiation): key j is visible to query i iff i - wl <= j <= i + wr.
  const int wl = GENERAL ? p.win_left : 0;
  const int wr = GENERAL ? p.win_right : 0;
  // Key blocks [first_blk(r), blocks_for(r)) of the 128-row tile starting at row r (empty past S).
  // Split-KV (general instantiation, kv_chunk > 0): the CTA's blockIdx.z
  // takes keys [kv_lo, kv_hi) only; kv_chunk is a multiple of 128.
  int kv_lo = 0, kv_hi = S;
  if constexpr (GENERAL) {
    if (p.kv_chunk > 0) {
      kv_lo = static_cast<int>(blockIdx.z) * p.kv_chunk;
      kv_hi = min(S, kv_lo + p.kv_chunk);
    }
  }
  auto first_blk = [&](int r) -> int {
    if constexpr (GENERAL) return r >= S ? 0 : max(kv_lo, r - wl) / kBlockN;
    else return 0;
  };
  auto blocks_for = [&](int r) -> int {
    if constexpr (GENERAL)
      return r >= S ? 0 : min((kv_hi + kBlockN - 1) / kBlockN, min(S - 1, r + kBlockM - 1 + wr) / kBlockN + 1);
    else return r >= S ? 0 : (p.causal ? min(n_kv, (r + kBlockM + kBlockN - 1) / kBlockN) : n_kv);
  };
  const int kb_cta = first_blk(row0);  // the CTA loads key blocks kb_cta, kb_cta + 1, ...
  // Tile t uses loaded blocks beg_t .. end_t - 1.
  const int lo0 = first_blk(row0) - kb_cta, hi0 = blocks_for(row0) - kb_cta;
  const int lo1 = first_blk(row0 + kBlockM) - kb_cta, hi1 = blocks_for(row0 + kBlockM) - kb_cta;
  const int beg0 = hi0 > lo0 ? lo0 : 0, end0 = hi0 > lo0 ? hi0 : 0;
  const int beg1 = hi1 > lo1 ? lo1 : 0, end1 = hi1 > lo1 ? hi1 : 0;
  const int nb0 = end0 - beg0;
  const int nb1 = end1 - beg1;
  const int nbp = max(end0, end1);  // blocks the CTA loads
  // TMA coordinates of `row` of `head` (x = column offset): (x, row, head) in
  // the {D, S, heads} maps, (x, head, tok0 + row) in the packed {D, heads, T} maps.
  auto tma_rows = [&](void* dst, const CUtensorMap* map, uint64_t* bar, int x, int row, int head) {
    if (GENERAL && packed)
      tma_load_3d(dst, map, bar, x, head, tok0 + row);
    else
      tma_load_3d(dst, map, bar, x, row, head);
  };

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < L::kStagesK; ++s) {
      mbar_init(&bar_kfull[s], 1);
      mbar_init(&bar_kempty[s], 2);  // released by both MMA warps
    }
    for (int s = 0; s < L::kStagesV; ++s) {
      mbar_init(&bar_vfull[s], 1);
      mbar_init(&bar_vempty[s], 2);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bar_sfull[t], 1);
      mbar_init(&bar_sfree[t], 4);  // one arrival per softmax warp
      mbar_init(&bar_pfull[t], 4);
      mbar_init(&bar_pvdone[t], 1);
      mbar_init(&bar_ofinal[t], 1);
    }
    mbar_init(&bar_drain[0], 1);
    mbar_init(&bar_drain[1], 1);
    for (int i = 0; i < 8; ++i) mbar_init(&bar_turn[i], 1);
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
            tma_rows(smem + L::kOffQ + t * L::kTileBytes + ch * L::kChunkBytes, &tm_q, bar_q,
                     ch * (L::kRowBytes / 2), row0 + t * kBlockM, q_head);
        // K and V blocks, each as two 64-row half-block copies.
        constexpr int kHalfBytes = (kBlockN / 2) * L::kRowBytes;
        // nk, nv: K and V blocks whose copies were started.
        int nk = 0, nv = 0;
        for (; nv < nbp; ++nv) {
          const int sk = nk % L::kStagesK;
          const int uk = nk / L::kStagesK;
          if (uk > 0 && !mbar_wait(&bar_kempty[sk], (uk - 1) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutLoad)) break;
          mbar_arrive_expect_tx(&bar_kfull[sk], L::kTileBytes);
#pragma unroll
          for (int ch = 0; ch < L::kChunks; ++ch)
#pragma unroll
            for (int h = 0; h < 2; ++h)
              tma_rows(smem + L::kOffK + sk * L::kTileBytes + ch * L::kChunkBytes + h * kHalfBytes, &tm_k,
                       &bar_kfull[sk], ch * (L::kRowBytes / 2), (kb_cta + nk) * kBlockN + h * (kBlockN / 2), kvh);
          ++nk;
          const int sv = nv % L::kStagesV;
          const int uv = nv / L::kStagesV;
          if (uv > 0 && !mbar_wait(&bar_vempty[sv], (uv - 1) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutLoad)) break;
          mbar_arrive_expect_tx(&bar_vfull[sv], L::kTileBytes);
#pragma unroll
          for (int ch = 0; ch < L::kChunks; ++ch)
#pragma unroll
            for (int h = 0; h < 2; ++h)
              tma_rows(smem + L::kOffV + sv * L::kTileBytes + ch * L::kChunkBytes + h * kHalfBytes, &tm_v,
                       &bar_vfull[sv], ch * (L::kRowBytes / 2), (kb_cta + nv) * kBlockN + h * (kBlockN / 2), kvh);
        }
        // Teardown: every copy this thread started must land before the CTA
        // exits (older copies of a ring were consumed before their stage was
        // reused).
        drain_wait(bar_q, 0, p.err);
        for (int x = (nk > L::kStagesK ? nk - L::kStagesK : 0); x < nk; ++x)
          drain_wait(&bar_kfull[x % L::kStagesK], (x / L::kStagesK) & 1, p.err);
        for (int x = (nv > L::kStagesV ? nv - L::kStagesV : 0); x < nv; ++x)
          drain_wait(&bar_vfull[x % L::kStagesV], (x / L::kStagesV) & 1, p.err);
      }
    } else if (warp == 9 || warp == 10) {
      // ------------------------------------------------------------ MMA issuers
      // Warp 9 issues tile 0's MMAs, warp 10 tile 1's, so one warp's commits
      // and barrier waits overlap the other's MMAs.  Each warp runs its code
      // converged and one elected lane issues each MMA; descriptors are built
      // once per stage and advanced by compile-time offsets.
      const int t = warp - 9;
      const int beg = t == 0 ? beg0 : beg1;  // this tile's loaded blocks beg .. nbt - 1
      const int nbt = t == 0 ? end0 : end1;
      constexpr uint32_t idesc_qk = make_idesc_f16(BF16, 128, kBlockN, false, false);
      constexpr uint32_t idesc_pv = make_idesc_f16(BF16, 128, D, false, true);
      const AccFlags acc = runtime_flags(S);
      const uint64_t q_desc = make_sdesc(sQ + t * L::kTileBytes, 16, 8 * L::kRowBytes, L::kSwz);
      // S_t = Q_t K(j)^T (the tile's block jl); with separate P, first wait
      // until the warpgroup has loaded S_t(jl-1).
      auto qk = [&](int j, int jl) -> bool {
        if (L::kSepP && jl > 0 && !warp_wait(&bar_sfree[t], (jl - 1) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutMma))
          return false;
        tc_fence_after();
        const uint64_t k_desc =
            make_sdesc(sK + (j % L::kStagesK) * L::kTileBytes, 16, 8 * L::kRowBytes, L::kSwz);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss_warp(tmem + L::kColS + 128u * t, desc_plus(q_desc, kmajor_step_bytes<D>(kk)),
                      desc_plus(k_desc, kmajor_step_bytes<D>(kk)), idesc_qk, kk > 0 ? acc.on : acc.off);
        mma_commit_warp(&bar_sfull[t]);
        return true;
      };
      // O_t += P_t(jl) V(j) once P_t(jl) is stored and O_t rescaled.
      auto pv = [&](int j, int jl) -> bool {
        const int st = j % L::kStagesV;
        if (!warp_wait(&bar_pfull[t], jl & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutMma)) return false;
        if (!warp_wait(&bar_vfull[st], (j / L::kStagesV) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutMma)) return false;
        tc_fence_after();
        const uint64_t v_desc = make_sdesc(sV + st * L::kTileBytes, L::kChunkBytes, 8 * L::kRowBytes, L::kSwz);
        const uint32_t t_p = tmem + L::kColP + L::kStrideP * t;
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk)
          mma_ts_warp(tmem + L::kColO + D * t, t_p + kk * 8, desc_plus(v_desc, mnmajor_step_bytes<D>(kk)), idesc_pv,
                      (jl > 0 || kk > 0) ? acc.on : acc.off);
        if (L::kSepP) mma_commit_warp(&bar_pvdone[t]);
        if (j == nbt - 1) mma_commit_warp(&bar_ofinal[t]);
        return true;
      };
      // This warp is done with V(x) once it has landed and its P V on it is
      // issued: it releases the stage (the arrival comes when the MMAs end).
      auto release_v = [&](int x) -> bool {
        const int st = x % L::kStagesV;
        if (!warp_wait(&bar_vfull[st], (x / L::kStagesV) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutMma)) return false;
        mma_commit_warp(&bar_vempty[st]);
        return true;
      };
      bool ok = warp_wait(bar_q, 0, abort_flag, p.err, p.wait_ns, kErrTimeoutMma);
      for (int j = 0; ok && j < nbp; ++j) {
        const int sk = j % L::kStagesK;
        ok = warp_wait(&bar_kfull[sk], (j / L::kStagesK) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutMma);
        if (!ok) break;
        tc_fence_after();
        const bool q_in = j >= beg && j < nbt;              // S_t of loaded block j
        const bool p_in = j >= 1 && j - 1 >= beg && j - 1 < nbt;  // P_t V of loaded block j - 1
        if (L::kSepP) {  // S_t(j) first, then O_t += P_t(j-1) V(j-1)
          if (q_in && !(ok = qk(j, j - beg))) break;
          mma_commit_warp(&bar_kempty[sk]);
          if (p_in && !(ok = pv(j - 1, j - 1 - beg))) break;
          if (j >= 1 && !(ok = release_v(j - 1))) break;
        } else {  // P_t(j-1) lives in S_t: its P V must precede S_t(j)
          if (p_in && !(ok = pv(j - 1, j - 1 - beg))) break;
          if (j >= 1 && !(ok = release_v(j - 1))) break;
          if (q_in && !(ok = qk(j, j - beg))) break;
          mma_commit_warp(&bar_kempty[sk]);  // K(j): this warp's score products on it are issued
        }
      }
      if (ok && nbp - 1 >= beg && nbp - 1 < nbt) ok = pv(nbp - 1, nbp - 1 - beg);
      if (ok && nbp > 0) release_v(nbp - 1);  // (split-KV: a CTA may load no block)
      // Teardown: wait for every MMA this warp issued.
      mma_commit_warp(&bar_drain[t]);
      drain_wait(&bar_drain[t], 0, p.err);
    }
  } else {
    regs_increase<kRegsHigh>();
    // ------------------------------------------------------------ softmax warpgroups
    const int t = warp >> 2;            // tile
    const int q4 = warp & 3;            // lane quarter (and SM sub-partition) of this warp
    const int r = threadIdx.x & 127;    // row within the tile == TMEM lane
    const int tile_row0 = row0 + t * kBlockM;
    const int row_g = tile_row0 + r;
    const int nb = t == 0 ? nb0 : nb1;
    const int nb_other = t == 0 ? nb1 : nb0;
    const int kb0 = kb_cta + (t == 0 ? beg0 : beg1);  // the tile's first key block
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t t_s = tmem + lane_base + L::kColS + 128u * t;
    const uint32_t t_p = tmem + lane_base + L::kColP + L::kStrideP * t;
    const uint32_t t_o = tmem + lane_base + L::kColO + D * t;
    const float sl2 = p.scale_log2;
    const float2 c2 = make_float2(sl2, sl2);
    const bool neg_scale = sl2 < 0.f;
    // Last (and, general instantiation, first) visible key of this row.
    const int last = GENERAL ? min(S - 1, row_g + wr) : (p.causal ? min(S - 1, row_g) : S - 1);
    const int first_key = row_g - wl;
    float m = -INFINITY;  // running (possibly stale) maximum, base-2 scaled
    float l = 0.f;
    bool alive = true;
    for (int j = 0; j < nb && alive; ++j) {
      uint32_t sr[kBlockN];
      if (!warp_wait(&bar_sfull[t], j & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutSoftmax)) {
        alive = false;
        break;
      }
      tc_fence_after();
      tmem_ld128(t_s, sr);
      if (L::kSepP) warp_arrive(&bar_sfree[t]);  // S_t(j) is in registers: the MMA may overwrite it
      const int kv0 = (kb0 + j) * kBlockN;
      const int lim = last - kv0;      // columns c <= lim are visible to this row
      const int lo = first_key - kv0;  // and (general instantiation) c >= lo
      // Masked blocks: the diagonal block under the causal mask (an edge of
      // the window band), and a ragged last key block.
      const bool masked = GENERAL ? (kv0 + kBlockN > S) || (kv0 + kBlockN - 1 > tile_row0 + wr) ||
                                        (kv0 < tile_row0 + kBlockM - 1 - wl)
                                  : (kv0 + kBlockN > S) || (p.causal && kv0 + kBlockN - 1 > tile_row0);
      if (j == 0) m = block_max_scaled<kBlockN, GENERAL>(sr, masked, lo, lim, sl2, neg_scale);
      // The two tiles' warps of one sub-partition take turns at the
      // exponentials, so one's loads, stores and waits overlap the other's.
      if (kTurns && (t == 0 ? j >= 1 && j - 1 < nb_other : j < nb_other) &&
          !warp_wait(&bar_turn[t * 4 + q4], (t == 0 ? j - 1 : j) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutSoftmax)) {
        alive = false;
        break;
      }
      uint32_t pk[kBlockN / 2];
      float alpha = 1.f;
      bool upd = false;
      float blk = exp_block<BF16, GENERAL>(sr, c2, m, masked, lo, lim, pk);
      // Every P~ <= 2^8 holds if the block's sum does.  Otherwise (or on NaN)
      // this block's maximum is too far above the stale m: move m to it,
      // rescale, and redo the block ("T5 讲解" §④ online update).  A window can
      // hide every key of a row's first blocks: the first block that shows the
      // row a key then sets m.
      bool need = !(blk <= kSumLimit);
      if constexpr (GENERAL) need = need || (m == -INFINITY && max(lo, 0) <= min(lim, kBlockN - 1));
      if (__any_sync(0xffffffffu, need)) {
        const float m_blk = block_max_scaled<kBlockN, GENERAL>(sr, masked, lo, lim, sl2, neg_scale);
        if (need && m_blk > m) {
          alpha = ex2(m - m_blk);
          m = m_blk;
          upd = true;
        }
        if (__any_sync(0xffffffffu, upd)) blk = exp_block<BF16, GENERAL>(sr, c2, m, masked, lo, lim, pk);
      }
      if (kTurns && (t == 0 ? j < nb_other : j + 1 < nb_other)) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_turn[(1 - t) * 4 + q4]);
      }
      l = l * alpha + blk;
      // With separate P, P_t(j-1) V(j-1) must be done before P_t is rewritten
      // and before O_t is rescaled.  (With P over S, S_t(j) being ready already
      // implies it: its commit covers the earlier P V.)
      if (L::kSepP && j > 0 && !warp_wait(&bar_pvdone[t], (j - 1) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutSoftmax)) {
        alive = false;
        break;
      }
      tc_fence_after();
      if (__any_sync(0xffffffffu, upd)) {
        // O holds the blocks before j relative to the old m: rescale this warp's rows.
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
      tmem_st32(t_p, pk);
      tmem_st32(t_p + 32, pk + 32);
      tmem_st_wait();
      warp_arrive(&bar_pfull[t]);
    }
    // ------------------------------------------------------------ epilogue
    const bool have = alive && nb > 0 && warp_wait(&bar_ofinal[t], 0, abort_flag, p.err, p.wait_ns, kErrTimeoutSoftmax);
    if (GENERAL && p.o_part != nullptr) {
      // Split-KV partial of shard blockIdx.z: fp32 O / l and L into
      // [shard][B*H*S] rows; a row that sees no key of the shard gets O = 0,
      // L = -inf (it then carries no weight in the merge).
      if (alive) {
        if (have) tc_fence_after();
        const bool row_ok = row_g < S;
        const bool seen = have && l > 0.f;
        const size_t prow = (static_cast<size_t>(blockIdx.z) * gridDim.x + bh) * S + (row_ok ? row_g : 0);
        float* orow = p.o_part + prow * D;
        const float inv_l = seen ? 1.f / l : 0.f;
#pragma unroll
        for (int c = 0; c < D; c += 16) {
          uint32_t o16[16];
          if (have) tmem_ld16(t_o + c, o16);
#pragma unroll
          for (int i = 0; i < 16; ++i) o16[i] = seen ? o16[i] : 0u;
          if (row_ok) store_row16_f32(orow + c, o16, inv_l);
        }
        if (row_ok) p.lse_part[prow] = seen ? (m + log2f(l)) * 0.69314718055994530942f : -INFINITY;
      }
    } else if (have) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      const bool row_ok = row_g < S;
      // Output row bh*S + row (fixed length) or (tok0 + row)*H + head (packed);
      // L at the same row, or at head*T + tok0 + row.
      const int rr = row_ok ? row_g : 0;
      const size_t o_row = (GENERAL && packed) ? static_cast<size_t>(tok0 + rr) * p.heads + q_head
                                               : static_cast<size_t>(bh) * S + rr;
      const size_t l_idx = (GENERAL && packed) ? static_cast<size_t>(q_head) * p.total + tok0 + rr : o_row;
      elem_t* orow = reinterpret_cast<elem_t*>(p.o) + o_row * D;
#pragma unroll
      for (int c = 0; c < D; c += 16) {
        uint32_t o16[16];
        tmem_ld16(t_o + c, o16);
        if (row_ok) store_row16<BF16>(orow + c, o16, inv_l);
      }
      if (row_ok) p.lse[l_idx] = (m + log2f(l)) * 0.69314718055994530942f;
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
template <int D, bool BF16, bool GENERAL>
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                         int BH, cudaStream_t stream) {
  using L = FwdLayout<D>;
  auto kern = fa_fwd_kernel<D, BF16, GENERAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
  if (e != cudaSuccess) return e;
  // The register split above assumes the launch gives exactly kLaunchRegs per
  // thread; with fewer, the softmax warpgroups' increase could never be met.
  cudaFuncAttributes attr;
  e = cudaFuncGetAttributes(&attr, kern);
  if (e != cudaSuccess) return e;
  if (attr.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
  // Split-KV: one grid slice per key shard.
  const int shards = (GENERAL && p.kv_chunk > 0) ? (p.S + p.kv_chunk - 1) / p.kv_chunk : 1;
  dim3 grid(BH, p.n_m_tiles, shards);
  kern<<<grid, kFwdThreads, L::kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_fwd(int D, bool bf16, bool general, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const FwdParams& p, int BH, cudaStream_t stream) {
#define FA_FWD_CASE(DD)                                                               \
  case DD:                                                                            \
    if (general)                                                                      \
      return bf16 ? launch_fwd_t<DD, true, true>(tq, tk, tv, p, BH, stream)           \
                  : launch_fwd_t<DD, false, true>(tq, tk, tv, p, BH, stream);         \
    return bf16 ? launch_fwd_t<DD, true, false>(tq, tk, tv, p, BH, stream)            \
                : launch_fwd_t<DD, false, false>(tq, tk, tv, p, BH, stream);
  switch (D) {
    case 16:
    case 32:
    case 64:
      return launch_fwd4(D, bf16, general, tq, tk, tv, p, BH, stream);
    FA_FWD_CASE(128)
    default:
      return cudaErrorInvalidValue;
  }
#undef FA_FWD_CASE
}

}  // namespace fa
