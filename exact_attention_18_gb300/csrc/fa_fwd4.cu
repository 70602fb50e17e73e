// Forward kernel for head dimensions D <= 64: exact attention with an online
// softmax, FlashAttention-2 loop order (query block outer, key/value block
// inner), on tcgen05 tensor cores with accumulators in tensor memory (TMEM).
//
// At D <= 64 a key block costs the tensor core as little as the softmax costs
// the exponential unit, so the kernel is built to keep that unit busy: one CTA
// per (batch*head, 512 query rows) = four 128-row query tiles, each with its
// own softmax warpgroup (thread = query row = TMEM lane, the split-Q partition
// of "Inside FlashAttention" §4.3), so every SM sub-partition holds four
// softmax warps whose loads, stores and waits hide behind each other's
// exponentials.  Key/value blocks are 64 rows.  Warp roles (640 threads):
//   warps 0-15  softmax: warp w serves tile w/4, TMEM lanes 32(w%4)..+31;
//   warp 16     TMA producer: the four Q tiles once, then K and V blocks
//               through a ring of shared-memory stages;
//   warps 17-18 MMA issuers, for tiles {0, 1} and {2, 3};
//   warp 19     idle (warps 16-19 give registers to the softmax warps).
//
// TMEM (512 columns): tile t owns columns [128t, 128t+128): S_t in the first
// 64 (fp32 scores of one block), O_t in the next D.  The 16-bit P_t(j) is
// written over the first 32 columns of S_t(j) and is the A operand of
// O_t += P_t V(j) straight from TMEM.  Per tile the MMA warp issues
//   O_t += P_t(j) V(j), then S_t = Q_t K(j+1)^T, then one commit,
// so "S_t(j+1) computed" also means "P_t(j) read and O_t updated": the softmax
// warps need one barrier wait per block, and they may rescale O_t as soon as
// they see S_t(j+1).
//
// Per key block j, per row, in the base-2 domain (c = scale * log2 e):
//   P~ = exp2(c * S_j - m),  l = alpha * l + rowsum(P~),  O += P~ V_j
// ("第二部分" §安全 / 在线 softmax; "fa-triton" Steps 2-4).  m is the exact
// maximum of the first block and is then kept, stale, for as long as a
// block's P~ sum stays <= 2^8 (so every P~ <= 2^8, far inside the 16-bit
// range); a block that breaks the bound moves m to its own maximum, rescales
// l and O by alpha = exp2(m_old - m) and is redone ("T5 讲解" §④ online update;
// "Inside FlashAttention" §4.1, fewer non-matmul operations).  Exact in real
// arithmetic.  Epilogue: O / l and L = (m + log2 l) ln 2.
//
// Causal: tile t visits key blocks up to its diagonal ("T5 讲解" §⑤); the
// element-wise mask runs only on the two blocks that cross the diagonal and
// on a ragged last block ("fa-triton" §Causal Mask 的处理：off-band 与 on-band).
//
// Fixed-length calls of up to 6144 rows run the persistent two-pipeline
// kernel of fa_fwd4p.cu instead, whose fixed cost per 256 rows is lower.
//
// GENERAL = true is the instantiation for packed variable-length batches and
// sliding windows ("Inside FlashAttention" §6.1): the CTA finds its sample
// from cu_seqlens, reads rows through {D, heads, T} tensor maps, and a tile
// visits only the key blocks that meet its band [i - win_left, i + win_right];
// blocks crossing either edge of the band are masked element-wise on both
// sides.  GENERAL = false is the fixed-length full/causal kernel, kept free of
// that bookkeeping.
#include "fa_softmax.cuh"

namespace fa {
using namespace ptx;

namespace {

constexpr int kF4Tiles = 4;
constexpr int kF4BlockN = 64;     // keys per block
constexpr int kF4RowsPerCta = kF4Tiles * kBlockM;
constexpr int kF4Producer = 16;
constexpr int kF4MmaWarp0 = 17;
// MMA issuers: warp kF4MmaWarp0 + w serves tiles w * kF4TilesPerMma, ...
// Measured at D = 64: one warp for all four tiles cannot keep the tensor core
// fed (each of its MMAs waits behind the last), four (one per tile) cost the
// softmax warps registers and issue slots; two were fastest.
constexpr int kF4MmaWarps = 2;
constexpr int kF4TilesPerMma = kF4Tiles / kF4MmaWarps;
// Whole warpgroups after the 16 softmax warps: producer + MMA warps + idle.
constexpr int kF4Threads = 512 + 128 * ((1 + kF4MmaWarps + 3) / 4);
// Register split: the launch gives every thread kF4LaunchRegs; the warps
// after the softmax warps drop to kF4RegsLow and the softmax warps rise to
// kF4RegsHigh.
constexpr int kF4LaunchRegs = kF4Threads == 640 ? 96 : 80;
constexpr uint32_t kF4RegsHigh = kF4Threads == 640 ? 104 : 96;
constexpr uint32_t kF4RegsLow = kF4Threads == 640 ? 64 : 48;
static_assert(512 * kF4RegsHigh + (kF4Threads - 512) * kF4RegsLow <= kF4Threads * kF4LaunchRegs, "register split");
constexpr float kF4SumLimit = 256.0f;
// Measured causal fp16 D = 64 forwards (us), persistent two-pipeline kernel / this one:
// S 1024 (B8 H16) 35.5 / 37.5, S 2048 (B4 H16) 46.3 / 50.9, S 4096 (B4 H16) 128.7 / 133.8,
// S 8192 (B2 H16) 232.0 / 226.5, S 16384 (B1 H16) 437 / 422.6.
constexpr int kPersistentMaxS = 6144;

template <int D, bool GENERAL>
struct F4Layout {
  static_assert(D <= 64, "four-tile forward is for D <= 64");
  using GQ = TileGeom<D, 128>;
  using GK = TileGeom<D, kF4BlockN>;
  // The general instantiation's tiles may run through blocks up to 6 apart
  // (window bands of consecutive 128-row tiles start 2 blocks apart), so it
  // keeps 8 stages in flight.
  static constexpr int kStages = (D <= 32 || GENERAL) ? 8 : 5;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kF4Tiles * GQ::kTileBytes;
  static constexpr int kOffV = kOffK + kStages * GK::kTileBytes;
  static constexpr int kOffBar = kOffV + kStages * GK::kTileBytes;
  // q, kfull[S], vfull[S], empty[S], sfull[4], pfull[4], ofinal[4], drain[MMA warps]
  static constexpr int kNumBars = 1 + 3 * kStages + 12 + kF4MmaWarps;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemUsed = kOffMisc + 16;
  // TMEM is allocated whole (512 columns): the shared-memory request keeps it
  // to one CTA per SM.
  static constexpr int kSmemBytes = (kSmemUsed + 1024) > 116 * 1024 ? (kSmemUsed + 1024) : 116 * 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 64;  // O_t at 128 t + 64; S_t (and P_t) at 128 t
  static_assert(kColO + D <= 128, "TMEM layout");
};

}  // namespace

// tm_q: 128-row boxes (the CTA's query tiles); tm_k, tm_v: 64-row boxes.
template <int D, bool BF16, bool GENERAL>
__global__ void __launch_bounds__(kF4Threads, 1)
    fa_fwd4_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using L = F4Layout<D, GENERAL>;
  using GQ = typename L::GQ;
  using GK = typename L::GK;
  using elem_t = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  constexpr int kBN = kF4BlockN;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* bar_q = bars;
  uint64_t* bar_kfull = bars + 1;
  uint64_t* bar_vfull = bar_kfull + L::kStages;
  uint64_t* bar_empty = bar_vfull + L::kStages;
  uint64_t* bar_sfull = bar_empty + L::kStages;  // [4] S_t(j) computed (and P_t(j-1) V(j-1) done)
  uint64_t* bar_pfull = bar_sfull + kF4Tiles;     // [4] P_t(j) stored, O_t rescaled
  uint64_t* bar_ofinal = bar_pfull + kF4Tiles;    // [4] last P V of tile t done
  uint64_t* bar_drain = bar_ofinal + kF4Tiles;    // one per MMA warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);

  const int warp = warp_index();
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
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
  const int cta = p.causal ? p.n_m_tiles - 1 - static_cast<int>(blockIdx.y) : static_cast<int>(blockIdx.y);
  const int row0 = cta * kF4RowsPerCta;
  if constexpr (GENERAL) {
    if (row0 >= S) return;  // packed batch: this CTA lies past its sample
  }
  const int n_kv = (S + kBN - 1) / kBN;
  // Window (general instantiation): key j is visible to query i iff i - wl <= j <= i + wr.
  const int wl = GENERAL ? p.win_left : 0;
  const int wr = GENERAL ? p.win_right : 0;
  // Key blocks [first_blk(r), blocks_for(r)) of the 128-row tile starting at
  // row r (empty past S).
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
    if constexpr (GENERAL) return r >= S ? 0 : max(kv_lo, r - wl) / kBN;
    else return 0;
  };
  auto blocks_for = [&](int r) -> int {
    if constexpr (GENERAL) return r >= S ? 0 : min((kv_hi + kBN - 1) / kBN, min(S - 1, r + kBlockM - 1 + wr) / kBN + 1);
    else return r >= S ? 0 : (p.causal ? min(n_kv, (r + kBlockM + kBN - 1) / kBN) : n_kv);
  };
  const int kb_cta = first_blk(row0);  // the CTA loads key blocks kb_cta, kb_cta + 1, ...
  int nbp = 0;                         // blocks the CTA loads
#pragma unroll
  for (int t = 0; t < kF4Tiles; ++t) nbp = max(nbp, blocks_for(row0 + t * kBlockM) - kb_cta);
  // TMA coordinates of `row` of `head`: (row, head) in the {D, S, heads}
  // maps, (head, tok0 + row) in the packed {D, heads, T} maps.
  auto tma_rows = [&](void* dst, const CUtensorMap* map, uint64_t* bar, int row, int head) {
    if (GENERAL && packed)
      tma_load_3d(dst, map, bar, 0, head, tok0 + row);
    else
      tma_load_3d(dst, map, bar, 0, row, head);
  };

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(&bar_kfull[s], 1);
      mbar_init(&bar_vfull[s], 1);
      mbar_init(&bar_empty[s], kF4MmaWarps);  // released by every MMA warp
    }
    for (int t = 0; t < kF4Tiles; ++t) {
      mbar_init(&bar_sfull[t], 1);
      mbar_init(&bar_pfull[t], 4);  // one arrival per softmax warp of the tile
      mbar_init(&bar_ofinal[t], 1);
    }
    for (int w = 0; w < kF4MmaWarps; ++w) mbar_init(&bar_drain[w], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kF4MmaWarp0) {
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

  if (warp >= kF4Producer) {
    regs_decrease<kF4RegsLow>();
    if (warp == kF4Producer) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        mbar_arrive_expect_tx(bar_q, kF4Tiles * GQ::kTileBytes);
#pragma unroll
        for (int t = 0; t < kF4Tiles; ++t)
          tma_rows(smem + L::kOffQ + t * GQ::kTileBytes, &tm_q, bar_q, row0 + t * kBlockM, q_head);
        int it = 0;
        for (; it < nbp; ++it) {
          const int st = it % L::kStages;
          const int use = it / L::kStages;
          if (use > 0 && !mbar_wait(&bar_empty[st], (use - 1) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutLoad)) break;
          mbar_arrive_expect_tx(&bar_kfull[st], GK::kTileBytes);
          tma_rows(smem + L::kOffK + st * GK::kTileBytes, &tm_k, &bar_kfull[st], (kb_cta + it) * kBN, kvh);
          mbar_arrive_expect_tx(&bar_vfull[st], GK::kTileBytes);
          tma_rows(smem + L::kOffV + st * GK::kTileBytes, &tm_v, &bar_vfull[st], (kb_cta + it) * kBN, kvh);
        }
        // Teardown: every copy this thread started must land before the CTA exits.
        drain_wait(bar_q, 0, p.err);
        for (int x = (it > L::kStages ? it - L::kStages : 0); x < it; ++x) {
          const int st = x % L::kStages;
          drain_wait(&bar_kfull[st], (x / L::kStages) & 1, p.err);
          drain_wait(&bar_vfull[st], (x / L::kStages) & 1, p.err);
        }
      }
    } else if (warp >= kF4MmaWarp0 && warp < kF4MmaWarp0 + kF4MmaWarps) {
      // ------------------------------------------------------------ MMA issuers
      // Warp kF4MmaWarp0 + w serves tiles w * kF4TilesPerMma, ... (a contiguous
      // pair).  Each runs converged and one elected lane issues every MMA.
      const int w = warp - kF4MmaWarp0;
      // Tile h of this warp uses loaded blocks beg[h] .. nbt[h]-1 (beg = 0
      // unless a window starts the tile's band later).
      int beg[kF4TilesPerMma], nbt[kF4TilesPerMma];
      int nbw = 0;
#pragma unroll
      for (int h = 0; h < kF4TilesPerMma; ++h) {
        const int r = row0 + (w * kF4TilesPerMma + h) * kBlockM;
        const int lo = first_blk(r) - kb_cta, hi = blocks_for(r) - kb_cta;
        beg[h] = hi > lo ? lo : 0;
        nbt[h] = hi > lo ? hi : 0;
        nbw = max(nbw, nbt[h]);
      }
      constexpr uint32_t idesc_qk = make_idesc_f16(BF16, 128, kBN, false, false);
      constexpr uint32_t idesc_pv = make_idesc_f16(BF16, 128, D, false, true);
      const AccFlags acc = runtime_flags(S);
      // S_t = Q_t K(j)^T into tile t's S columns.
      auto qk = [&](int t, int j) {
        const uint64_t q_desc = make_sdesc(sQ + t * GQ::kTileBytes, 16, 8 * GQ::kRowBytes, GQ::kSwz);
        const uint64_t k_desc = make_sdesc(sK + (j % L::kStages) * GK::kTileBytes, 16, 8 * GK::kRowBytes, GK::kSwz);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss_warp(tmem + 128u * t, desc_plus(q_desc, kmajor_step_bytes<D, 128>(kk)),
                      desc_plus(k_desc, kmajor_step_bytes<D, kBN>(kk)), idesc_qk, kk > 0 ? acc.on : acc.off);
      };
      // O_t += P_t(j) V(j), P from tile t's S columns; jl = the tile's own block count so far.
      auto pv = [&](int t, int j, int jl) {
        const uint64_t v_desc =
            make_sdesc(sV + (j % L::kStages) * GK::kTileBytes, GK::kChunkBytes, 8 * GK::kRowBytes, GK::kSwz);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ts_warp(tmem + 128u * t + L::kColO, tmem + 128u * t + kk * 8,
                      desc_plus(v_desc, mnmajor_step_bytes<D>(kk)), idesc_pv, (jl > 0 || kk > 0) ? acc.on : acc.off);
      };
      if constexpr (GENERAL) {
        // Each tile runs through its own blocks beg[h] .. nbt[h]-1 one step at a
        // time, so under a window band (tiles' bands shifted by 128 rows) every
        // tile is busy at every step instead of waiting while the CTA streams
        // blocks outside its band.  The warp releases a block's stage after the
        // last of its tiles to use it has issued its P V (a tile whose band
        // starts earlier uses a block at a later step; at the same step, the
        // tile issued last), and releases blocks neither tile uses once they
        // have landed.
        bool ok = warp_wait(bar_q, 0, abort_flag, p.err, p.wait_ns, kErrTimeoutMma);
        int n[kF4TilesPerMma];
        int nsteps = 0, lo_used = nbp, hi_used = 0;
#pragma unroll
        for (int h = 0; h < kF4TilesPerMma; ++h) {
          n[h] = nbt[h] - beg[h];
          nsteps = max(nsteps, n[h]);
          if (n[h] > 0) {
            lo_used = min(lo_used, beg[h]);
            hi_used = max(hi_used, nbt[h]);
          }
        }
        if (hi_used == 0) lo_used = 0;
        auto release_landed = [&](int x) {  // a block this warp does not use
          const int sx = x % L::kStages;
          ok = ok && warp_wait(&bar_vfull[sx], (x / L::kStages) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutMma) &&
               warp_wait(&bar_kfull[sx], (x / L::kStages) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutMma);
          if (ok) mma_commit_warp(&bar_empty[sx]);
        };
        for (int x = 0; ok && x < lo_used; ++x) release_landed(x);
#pragma unroll
        for (int h = 0; h < kF4TilesPerMma; ++h) {
          if (!ok || n[h] <= 0) continue;
          const int x = beg[h];
          ok = warp_wait(&bar_kfull[x % L::kStages], (x / L::kStages) & 1, abort_flag, p.err, p.wait_ns,
                         kErrTimeoutMma);
          if (!ok) break;
          tc_fence_after();
          qk(w * kF4TilesPerMma + h, x);
          mma_commit_warp(&bar_sfull[w * kF4TilesPerMma + h]);
        }
        for (int k = 0; ok && k < nsteps; ++k) {
#pragma unroll
          for (int h = 0; h < kF4TilesPerMma; ++h) {
            if (!ok) break;
            if (k >= n[h]) continue;
            const int t = w * kF4TilesPerMma + h;
            const int x = beg[h] + k;
            ok = warp_wait(&bar_vfull[x % L::kStages], (x / L::kStages) & 1, abort_flag, p.err, p.wait_ns,
                           kErrTimeoutMma);
            if (ok && k + 1 < n[h])
              ok = warp_wait(&bar_kfull[(x + 1) % L::kStages], ((x + 1) / L::kStages) & 1, abort_flag, p.err,
                             p.wait_ns, kErrTimeoutMma);
            ok = ok && warp_wait(&bar_pfull[t], k & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutMma);
            if (!ok) break;
            tc_fence_after();
            pv(t, x, k);
            if (k + 1 < n[h]) {
              qk(t, x + 1);
              mma_commit_warp(&bar_sfull[t]);
            } else {
              mma_commit_warp(&bar_ofinal[t]);
            }
            // The last of this warp's tiles to use block x releases it: a tile
            // whose band starts earlier uses a block at a later step.
            bool last_user = true;
#pragma unroll
            for (int e = 0; e < kF4TilesPerMma; ++e)
              if (e != h && beg[e] <= x && x < nbt[e] && x - beg[e] > k) last_user = false;
#pragma unroll
            for (int e = h + 1; e < kF4TilesPerMma; ++e)  // same step: the tile issued last releases
              if (beg[e] <= x && x < nbt[e] && x - beg[e] == k) last_user = false;
            if (last_user) mma_commit_warp(&bar_empty[x % L::kStages]);
          }
        }
        for (int x = hi_used; ok && x < nbp; ++x) release_landed(x);
      } else {
        bool ok = warp_wait(bar_q, 0, abort_flag, p.err, p.wait_ns, kErrTimeoutMma);
        if (ok && nbw > 0) ok = warp_wait(&bar_kfull[0], 0, abort_flag, p.err, p.wait_ns, kErrTimeoutMma);
        if (ok) {
          tc_fence_after();
  #pragma unroll
          for (int h = 0; h < kF4TilesPerMma; ++h) {
            if (nbt[h] == 0) continue;
            const int t = w * kF4TilesPerMma + h;
            qk(t, 0);
            mma_commit_warp(&bar_sfull[t]);
          }
        }
        int j = 0;
        for (; ok && j < nbw; ++j) {
          const int st = j % L::kStages;
          ok = warp_wait(&bar_vfull[st], (j / L::kStages) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutMma);
          // K(j+1) for the next score products (if a tile of this warp goes on).
          if (ok && j + 1 < nbw)
            ok = warp_wait(&bar_kfull[(j + 1) % L::kStages], ((j + 1) / L::kStages) & 1, abort_flag, p.err, p.wait_ns,
                           kErrTimeoutMma);
  #pragma unroll
          for (int h = 0; h < kF4TilesPerMma; ++h) {
            if (!ok) break;
            if (j >= nbt[h]) continue;
            const int t = w * kF4TilesPerMma + h;
            const int jl = j;
            ok = warp_wait(&bar_pfull[t], jl & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutMma);
            if (!ok) break;
            tc_fence_after();
            pv(t, j, jl);
            if (j + 1 < nbt[h]) {
              qk(t, j + 1);
              mma_commit_warp(&bar_sfull[t]);
            } else {
              mma_commit_warp(&bar_ofinal[t]);
            }
          }
          if (ok) mma_commit_warp(&bar_empty[st]);  // this warp's MMAs on K(j), V(j) are issued
        }
        // Blocks the CTA loads but no tile of this warp uses: release each once
        // it has landed (so the arrival counts toward the right phase).
        for (; ok && j < nbp; ++j) {
          const int st = j % L::kStages;
          ok = warp_wait(&bar_vfull[st], (j / L::kStages) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutMma) &&
               warp_wait(&bar_kfull[st], (j / L::kStages) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutMma);
          if (ok) mma_commit_warp(&bar_empty[st]);
        }
      }
      // Teardown: wait for every MMA this warp issued.
      mma_commit_warp(&bar_drain[w]);
      drain_wait(&bar_drain[w], 0, p.err);
    }
  } else {
    regs_increase<kF4RegsHigh>();
    // ------------------------------------------------------------ softmax warps
    const int t = warp >> 2;  // tile
    const int q4 = warp & 3;  // lane quarter
    const int r = q4 * 32 + lane;
    const int tile_row0 = row0 + t * kBlockM;
    const int row_g = tile_row0 + r;
    const int kb0 = first_blk(tile_row0);  // the tile's first key block
    const int nb = max(0, blocks_for(tile_row0) - kb0);
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t t_s = tmem + lane_base + 128u * t;  // S_t, and P_t over it
    const uint32_t t_o = t_s + L::kColO;
    const float sl2 = p.scale_log2;
    const float2 c2 = make_float2(sl2, sl2);
    const bool neg_scale = sl2 < 0.f;
    // Last (and, general instantiation, first) visible key of this row.
    const int last = GENERAL ? min(S - 1, row_g + wr) : (p.causal ? min(S - 1, row_g) : S - 1);
    const int first_key = row_g - wl;
    float m = -INFINITY;  // running (possibly stale) maximum, base-2 scaled
    float l = 0.f;
    bool alive = true;
    for (int j = 0; j < nb; ++j) {
      if (!warp_wait(&bar_sfull[t], j & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutSoftmax)) {
        alive = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[kBN];
      tmem_ld64(t_s, sr);
      const int kv0 = (kb0 + j) * kBN;
      const int lim = last - kv0;      // columns c <= lim are visible to this row
      const int lo = first_key - kv0;  // and (general instantiation) c >= lo
      // Masked blocks: those crossing the diagonal under the causal mask (an
      // edge of the window band), and a ragged last key block.
      const bool masked =
          GENERAL ? (kv0 + kBN > S) || (kv0 + kBN - 1 > tile_row0 + wr) || (kv0 < tile_row0 + kBlockM - 1 - wl)
                  : (kv0 + kBN > S) || (p.causal && kv0 + kBN - 1 > tile_row0);
      if (j == 0) m = block_max_scaled<kBN, GENERAL>(sr, masked, lo, lim, sl2, neg_scale);
      float alpha = 1.f;
      bool upd = false;
      float blk;
      // P~ of the block, written 16 keys at a time over the S columns just read.
      auto exps = [&]() {
        const float m_use = (m == -INFINITY) ? 0.f : m;  // rows with no visible key so far
        const float2 negm = make_float2(-m_use, -m_use);
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
        if (masked) {
#pragma unroll
          for (int k0 = 0; k0 < kBN; k0 += 16) {
            uint32_t pk[8];
            exp16<BF16, true, GENERAL>(sr, k0, c2, negm, lo, lim, acc, pk);
            tmem_st8(t_s + k0 / 2, pk);
          }
        } else {
#pragma unroll
          for (int k0 = 0; k0 < kBN; k0 += 16) {
            uint32_t pk[8];
            exp16<BF16, false>(sr, k0, c2, negm, lo, lim, acc, pk);
            tmem_st8(t_s + k0 / 2, pk);
          }
        }
        const float2 a = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
        return a.x + a.y;
      };
      blk = exps();
      // Every P~ <= 2^8 holds if the block's sum does.  Otherwise (or on NaN)
      // the stale m is too far below this block's maximum: move m, rescale,
      // and redo the block.
      bool need = !(blk <= kF4SumLimit);
      if constexpr (GENERAL) {
        // A window can hide every key of a row's first blocks: m is still
        // -inf there, and the first block that shows the row a key sets it.
        need = need || (m == -INFINITY && max(lo, 0) <= min(lim, kBN - 1));
      }
      if (__any_sync(0xffffffffu, need)) {
        const float m_blk = block_max_scaled<kBN, GENERAL>(sr, masked, lo, lim, sl2, neg_scale);
        if (need && m_blk > m) {
          alpha = ex2(m - m_blk);
          m = m_blk;
          upd = true;
        }
        if (__any_sync(0xffffffffu, upd)) {
          tmem_st_wait();  // the first pass's stores land before they are overwritten
          blk = exps();
          // O_t holds the blocks before j relative to the old m (P_t(j-1) V(j-1)
          // is complete: S_t(j) was committed after it).
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
      }
      l = l * alpha + blk;
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
  if (warp == kF4MmaWarp0) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

namespace {
template <int D, bool BF16, bool GENERAL>
cudaError_t launch_fwd4_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                          int BH, cudaStream_t stream) {
  using L = F4Layout<D, GENERAL>;
  auto kern = fa_fwd4_kernel<D, BF16, GENERAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
  if (e != cudaSuccess) return e;
  // The register split assumes the launch gives exactly kF4LaunchRegs per
  // thread; with fewer, the softmax warps' increase could never be met.
  cudaFuncAttributes attr;
  e = cudaFuncGetAttributes(&attr, kern);
  if (e != cudaSuccess) return e;
  if (attr.numRegs != kF4LaunchRegs) return cudaErrorInvalidConfiguration;
  // Split-KV: one grid slice per key shard.
  const int shards = (GENERAL && p.kv_chunk > 0) ? (p.S + p.kv_chunk - 1) / p.kv_chunk : 1;
  dim3 grid(BH, p.n_m_tiles, shards);
  kern<<<grid, kF4Threads, L::kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}
}  // namespace

int fwd_rows_per_cta(int D) { return D <= 64 ? kF4RowsPerCta : 2 * kBlockM; }

cudaError_t launch_fwd4(int D, bool bf16, bool general, const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv, const FwdParams& p, int BH, cudaStream_t stream) {
  // Fixed-length sequences up to kPersistentMaxS rows run the persistent
  // two-pipeline kernel (fa_fwd4p.cu), whose lower fixed cost per 256 rows
  // pays off there; longer ones this kernel, whose per-block cost is lower.
  if (!general && p.S <= kPersistentMaxS) return launch_fwd4p(D, bf16, tq, tk, tv, p, BH, stream);
#define FA_FWD4_CASE(DD)                                                                       \
  case DD:                                                                                     \
    if (general)                                                                               \
      return bf16 ? launch_fwd4_t<DD, true, true>(tq, tk, tv, p, BH, stream)                   \
                  : launch_fwd4_t<DD, false, true>(tq, tk, tv, p, BH, stream);                 \
    return bf16 ? launch_fwd4_t<DD, true, false>(tq, tk, tv, p, BH, stream)                    \
                : launch_fwd4_t<DD, false, false>(tq, tk, tv, p, BH, stream);
  switch (D) {
    FA_FWD4_CASE(16)
    FA_FWD4_CASE(32)
    FA_FWD4_CASE(64)
    default:
      return cudaErrorInvalidValue;
  }
#undef FA_FWD4_CASE
}

}  // namespace fa
