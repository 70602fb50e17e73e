// Forward kernel for head dimensions D <= 64 and fixed-length sequences of up
// to 6144 rows (launch_fwd4 picks it): persistent CTAs, each running two
// independent pipelines.
//
// The per-block work is that of the four-tile kernel (fa_fwd4.cu, whose
// header describes the softmax, the TMEM layout of a tile and the MMA order):
// 128-row query tiles, 64-key blocks, P written over S in TMEM, one commit per
// tile and block, a stale maximum kept while a block's sum stays <= 2^8.
// What differs is how the tiles are grouped.  A work item is 256 query rows
// of one head (two tiles), and each CTA runs two pipelines, each with its own
// Q buffer, K/V ring, producer warp, MMA warp and two softmax warpgroups, that
// walk through their own sequences of work items.  So
//   - the two tiles of an item differ by two key blocks under the causal mask
//     (four consecutive tiles differ by six, and a CTA's last tile ran those
//     six blocks with the SM partly idle);
//   - while one pipeline loads a new item's Q and first K/V blocks, or stores
//     its outputs, the other keeps the tensor core and the exponential unit
//     busy;
// at the cost of each pipeline streaming its own K and V (twice the four-tile
// kernel's shared-memory fills).
//
// Work items are ordered heaviest first under the causal mask (the items at
// the bottom of every head, then the next row up, ...) and dealt to the
// pipelines in a snake: round r gives item r*P + g to pipeline g when r is
// even and r*P + P-1-g when it is odd (P pipelines), which evens out the
// pipelines' total work without a device-side queue.
//
// Warp roles (640 threads):
//   warps 0-7    pipeline 0's softmax warps: tile 0 (warps 0-3), tile 1 (4-7);
//   warps 8-15   pipeline 1's: tile 2 (8-11), tile 3 (12-15);
//   warp 16      pipeline 0's TMA producer, warp 19 pipeline 1's;
//   warp 17      pipeline 0's MMA issuer, warp 18 pipeline 1's.
// Softmax warp w serves TMEM lanes 32(w%4).. of tile w/4; tile t owns TMEM
// columns [128t, 128t+128) (S, and P over it, then O), as in the four-tile
// kernel.
//
// Barrier phases run on across a pipeline's items: K/V stages by a running
// block count, S/P barriers by each tile's running block count, the Q and
// final-O barriers by item.  Q of the next item is loaded once the score
// products of the current item's last key block (the last reads of Q) are
// done; the first K/V blocks of the next item go out before that.
#include "fa_softmax.cuh"

namespace fa {
using namespace ptx;

namespace {

constexpr int kPTiles = 2;   // 128-row tiles per work item and pipeline
constexpr int kPPipes = 2;   // pipelines per CTA
constexpr int kPBlockN = 64; // keys per block
constexpr int kPRowsPerItem = kPTiles * kBlockM;
constexpr int kPThreads = 640;
constexpr int kPProducer0 = 16, kPMma0 = 17, kPMma1 = 18, kPProducer1 = 19;
// Register split as in the four-tile kernel: softmax warps 104, the others 64.
constexpr int kPLaunchRegs = 96;
constexpr uint32_t kPRegsHigh = 104;
constexpr uint32_t kPRegsLow = 64;
static_assert(512 * kPRegsHigh + 128 * kPRegsLow <= kPThreads * kPLaunchRegs, "register split");
constexpr float kPSumLimit = 256.0f;

template <int D>
struct FPLayout {
  static_assert(D <= 64, "persistent forward is for D <= 64");
  using GQ = TileGeom<D, 128>;
  using GK = TileGeom<D, kPBlockN>;
  // K/V blocks in flight per pipeline (at D = 64, five: 3 % faster than four at causal B1 H16
  // S16384, 1 % at B4 H16 S4096; the two pipelines then fill 225 of the 227 KB).
  static constexpr int kStages = D <= 32 ? 8 : 5;
  // Per pipeline: Q (two tiles), then the K ring, then the V ring.
  static constexpr int kOffK = kPTiles * GQ::kTileBytes;
  static constexpr int kOffV = kOffK + kStages * GK::kTileBytes;
  static constexpr int kPipeBytes = kOffV + kStages * GK::kTileBytes;
  static constexpr int kOffBar = kPPipes * kPipeBytes;
  // Per pipeline: q_full, q_empty, k_full[S], v_full[S], empty[S], s_full[2], p_full[2], o_final[2], drain.
  static constexpr int kBarsPerPipe = 2 + 3 * kStages + 3 * kPTiles + 1;
  static constexpr int kOffMisc = kOffBar + kPPipes * kBarsPerPipe * 8;
  static constexpr int kSmemUsed = kOffMisc + 16;
  static constexpr int kSmemBytes = kSmemUsed + 1024;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColO = 64;  // O_t at 128 t + 64; S_t (and P_t) at 128 t
  static_assert(kColO + D <= 128, "TMEM layout");
};

}  // namespace

// tm_q: 128-row boxes; tm_k, tm_v: 64-row boxes ({D, S, heads} maps).
// n_rb: 256-row items per head; n_items = B*H * n_rb.
template <int D, bool BF16>
__global__ void __launch_bounds__(kPThreads, 1)
    fa_fwd4p_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const FwdParams p, int n_items, int n_rb) {
  using L = FPLayout<D>;
  using GQ = typename L::GQ;
  using GK = typename L::GK;
  using elem_t = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  constexpr int kBN = kPBlockN;
  constexpr int kS = L::kStages;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);

  const int warp = warp_index();
  const int lane = threadIdx.x & 31;
  // This warp's pipeline and its shared memory and barriers.
  const int pipe = warp < 16 ? (warp >> 3) : (warp == kPProducer0 || warp == kPMma0 ? 0 : 1);
  uint8_t* pbase = smem + pipe * L::kPipeBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar) + pipe * L::kBarsPerPipe;
  uint64_t* bar_qfull = bars;           // Q of the pipeline's current item landed
  uint64_t* bar_qempty = bars + 1;      // the item's last score products (last reads of Q) done
  uint64_t* bar_kfull = bars + 2;       // [S]
  uint64_t* bar_vfull = bar_kfull + kS;  // [S]
  uint64_t* bar_empty = bar_vfull + kS;  // [S] stage's K, V read by every MMA that uses them
  uint64_t* bar_sfull = bar_empty + kS;  // [2] S_t(j) computed (and P_t(j-1) V(j-1) done)
  uint64_t* bar_pfull = bar_sfull + kPTiles;   // [2] P_t(j) stored, O_t rescaled
  uint64_t* bar_ofinal = bar_pfull + kPTiles;  // [2] last P V of the tile's item done
  uint64_t* bar_drain = bar_ofinal + kPTiles;

  const int S = p.S;
  const int n_kv = (S + kBN - 1) / kBN;
  const int BH = n_items / n_rb;
  // Item sequence of this pipeline (snake over the heaviest-first order).
  const int P = kPPipes * static_cast<int>(gridDim.x);
  const int g = static_cast<int>(blockIdx.x) * kPPipes + pipe;
  auto item_at = [&](int r) -> int {
    const int k = r * P + ((r & 1) ? (P - 1 - g) : g);
    return k < n_items ? k : -1;
  };
  // Item k: head bh, 256-row block rb (bottom rows first under the causal mask).
  auto decode = [&](int k, int* bh, int* rb) {
    const int q = k / BH;
    *bh = k - q * BH;
    *rb = p.causal ? n_rb - 1 - q : q;
  };
  // Key blocks of the 128-row tile starting at row r (0 past S).
  auto blocks_for = [&](int r) -> int {
    return r >= S ? 0 : (p.causal ? min(n_kv, (r + kBlockM + kBN - 1) / kBN) : n_kv);
  };

  if (threadIdx.x == 0) {
#pragma unroll
    for (int pp = 0; pp < kPPipes; ++pp) {
      uint64_t* b = reinterpret_cast<uint64_t*>(smem + L::kOffBar) + pp * L::kBarsPerPipe;
      mbar_init(&b[0], 1);
      mbar_init(&b[1], 1);
      for (int s = 0; s < kS; ++s) {
        mbar_init(&b[2 + s], 1);
        mbar_init(&b[2 + kS + s], 1);
        mbar_init(&b[2 + 2 * kS + s], 1);  // released by the pipeline's one MMA warp
      }
      for (int t = 0; t < kPTiles; ++t) {
        mbar_init(&b[2 + 3 * kS + t], 1);
        mbar_init(&b[2 + 3 * kS + kPTiles + t], 4);  // one arrival per softmax warp of the tile
        mbar_init(&b[2 + 3 * kS + 2 * kPTiles + t], 1);
      }
      mbar_init(&b[2 + 3 * kS + 3 * kPTiles], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kPMma0) {
    tmem_alloc(tmem_slot, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sQ = smem_u32(pbase);
  const uint32_t sK = smem_u32(pbase + L::kOffK);
  const uint32_t sV = smem_u32(pbase + L::kOffV);

  if (warp >= 16) {
    regs_decrease<kPRegsLow>();
    if (warp == kPProducer0 || warp == kPProducer1) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        if (pipe == 0) {
          prefetch_tmap(&tm_q);
          prefetch_tmap(&tm_k);
          prefetch_tmap(&tm_v);
        }
        bool ok = true;
        int it = 0;      // K/V blocks loaded so far (ring position)
        int n = 0;       // items whose Q load was issued
        for (int r = 0; ok; ++r) {
          const int k = item_at(r);
          if (k < 0) break;
          int bh, rb;
          decode(k, &bh, &rb);
          const int row0 = rb * kPRowsPerItem;
          const int kvh = bh / p.group;
          const int nbp = max(blocks_for(row0), blocks_for(row0 + kBlockM));
          // The item's first K/V blocks go out before its Q, whose buffer the
          // previous item may still be reading.
          const int pre = min(nbp, 2);
          auto load_kv = [&](int j) -> bool {
            const int st = it % kS;
            const int use = it / kS;
            if (use > 0 && !mbar_wait(&bar_empty[st], (use - 1) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutLoad))
              return false;
            mbar_arrive_expect_tx(&bar_kfull[st], GK::kTileBytes);
            tma_load_3d(pbase + L::kOffK + st * GK::kTileBytes, &tm_k, &bar_kfull[st], 0, j * kBN, kvh);
            mbar_arrive_expect_tx(&bar_vfull[st], GK::kTileBytes);
            tma_load_3d(pbase + L::kOffV + st * GK::kTileBytes, &tm_v, &bar_vfull[st], 0, j * kBN, kvh);
            ++it;
            return true;
          };
          for (int j = 0; ok && j < pre; ++j) ok = load_kv(j);
          if (ok && n > 0) ok = mbar_wait(bar_qempty, (n - 1) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutLoad);
          if (!ok) break;
          mbar_arrive_expect_tx(bar_qfull, kPTiles * GQ::kTileBytes);
#pragma unroll
          for (int t = 0; t < kPTiles; ++t)
            tma_load_3d(pbase + t * GQ::kTileBytes, &tm_q, bar_qfull, 0, row0 + t * kBlockM, bh);
          ++n;
          for (int j = pre; ok && j < nbp; ++j) ok = load_kv(j);
        }
        // Teardown: every copy this thread started must land before the CTA exits.
        if (n > 0) drain_wait(bar_qfull, (n - 1) & 1, p.err);
        for (int x = (it > kS ? it - kS : 0); x < it; ++x) {
          drain_wait(&bar_kfull[x % kS], (x / kS) & 1, p.err);
          drain_wait(&bar_vfull[x % kS], (x / kS) & 1, p.err);
        }
      }
    } else {
      // ------------------------------------------------------------ MMA issuer
      // Runs converged; one elected lane issues each MMA.  Tiles 2 pipe and
      // 2 pipe + 1, in that order at every block.
      const int t0 = kPTiles * pipe;
      constexpr uint32_t idesc_qk = make_idesc_f16(BF16, 128, kBN, false, false);
      constexpr uint32_t idesc_pv = make_idesc_f16(BF16, 128, D, false, true);
      const AccFlags acc = runtime_flags(S);
      auto qk = [&](int t, int st) {  // S_t = Q_t K(stage st)^T
        const uint64_t q_desc =
            make_sdesc(sQ + (t - t0) * GQ::kTileBytes, 16, 8 * GQ::kRowBytes, GQ::kSwz);
        const uint64_t k_desc = make_sdesc(sK + st * GK::kTileBytes, 16, 8 * GK::kRowBytes, GK::kSwz);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss_warp(tmem + 128u * t, desc_plus(q_desc, kmajor_step_bytes<D, 128>(kk)),
                      desc_plus(k_desc, kmajor_step_bytes<D, kBN>(kk)), idesc_qk, kk > 0 ? acc.on : acc.off);
      };
      auto pv = [&](int t, int st, int jl) {  // O_t += P_t V(stage st); jl = the block's index in the item
        const uint64_t v_desc = make_sdesc(sV + st * GK::kTileBytes, GK::kChunkBytes, 8 * GK::kRowBytes, GK::kSwz);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ts_warp(tmem + 128u * t + L::kColO, tmem + 128u * t + kk * 8,
                      desc_plus(v_desc, mnmajor_step_bytes<D>(kk)), idesc_pv, (jl > 0 || kk > 0) ? acc.on : acc.off);
      };
      bool ok = true;
      int it = 0;                 // K/V blocks consumed so far
      int n = 0;                  // items started
      int jt[kPTiles] = {0, 0};   // blocks per tile so far (P barrier phases)
      for (int r = 0; ok; ++r) {
        const int k = item_at(r);
        if (k < 0) break;
        int bh, rb;
        decode(k, &bh, &rb);
        const int row0 = rb * kPRowsPerItem;
        int nbt[kPTiles];
#pragma unroll
        for (int h = 0; h < kPTiles; ++h) nbt[h] = blocks_for(row0 + h * kBlockM);
        const int nbw = max(nbt[0], nbt[1]);  // >= 1: row0 < S
        ok = warp_wait(bar_qfull, n & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutMma) &&
             warp_wait(&bar_kfull[it % kS], (it / kS) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutMma);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < kPTiles; ++h) {
          if (nbt[h] == 0) continue;
          qk(t0 + h, it % kS);
          mma_commit_warp(&bar_sfull[h]);
        }
        if (nbw == 1) mma_commit_warp(bar_qempty);  // those were the item's last reads of Q
        for (int j = 0; ok && j < nbw; ++j) {
          const int x = it + j;
          const int st = x % kS;
          ok = warp_wait(&bar_vfull[st], (x / kS) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutMma);
          if (ok && j + 1 < nbw)
            ok = warp_wait(&bar_kfull[(x + 1) % kS], ((x + 1) / kS) & 1, abort_flag, p.err, p.wait_ns,
                           kErrTimeoutMma);
#pragma unroll
          for (int h = 0; h < kPTiles; ++h) {
            if (!ok) break;
            if (j >= nbt[h]) continue;
            ok = warp_wait(&bar_pfull[h], jt[h] & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutMma);
            if (!ok) break;
            tc_fence_after();
            pv(t0 + h, st, j);
            if (j + 1 < nbt[h]) {
              qk(t0 + h, (x + 1) % kS);
              mma_commit_warp(&bar_sfull[h]);
            } else {
              mma_commit_warp(&bar_ofinal[h]);
            }
            ++jt[h];
          }
          if (!ok) break;
          if (j + 2 == nbw) mma_commit_warp(bar_qempty);  // the last block's score products are issued
          mma_commit_warp(&bar_empty[st]);
        }
        it += nbw;
        ++n;
      }
      // Teardown: wait for every MMA this warp issued.
      mma_commit_warp(bar_drain);
      drain_wait(bar_drain, 0, p.err);
    }
  } else {
    regs_increase<kPRegsHigh>();
    // ------------------------------------------------------------ softmax warps
    const int h = (warp >> 2) & 1;    // tile within the item
    const int t = kPTiles * pipe + h;  // TMEM tile
    const int q4 = warp & 3;          // lane quarter
    const int rr = q4 * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t t_s = tmem + lane_base + 128u * t;  // S_t, and P_t over it
    const uint32_t t_o = t_s + L::kColO;
    const float sl2 = p.scale_log2;
    const float2 c2 = make_float2(sl2, sl2);
    const bool neg_scale = sl2 < 0.f;
    bool alive = true;
    int jg = 0;  // blocks of this tile so far (S barrier phases)
    int on = 0;  // items in which this tile had blocks (final-O barrier phases)
    for (int r = 0; alive; ++r) {
      const int k = item_at(r);
      if (k < 0) break;
      int bh, rb;
      decode(k, &bh, &rb);
      const int tile_row0 = rb * kPRowsPerItem + h * kBlockM;
      const int row_g = tile_row0 + rr;
      const int nb = blocks_for(tile_row0);
      if (nb == 0) continue;
      const int last = p.causal ? min(S - 1, row_g) : S - 1;  // last visible key of this row
      float m = -INFINITY;  // running (possibly stale) maximum, base-2 scaled
      float l = 0.f;
      for (int j = 0; j < nb; ++j, ++jg) {
        if (!warp_wait(&bar_sfull[h], jg & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutSoftmax)) {
          alive = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[kBN];
        tmem_ld64(t_s, sr);
        const int kv0 = j * kBN;
        const int lim = last - kv0;  // columns c <= lim are visible to this row
        // Masked blocks: those crossing the diagonal, and a ragged last key block.
        const bool masked = (kv0 + kBN > S) || (p.causal && kv0 + kBN - 1 > tile_row0);
        if (j == 0) m = block_max_scaled<kBN>(sr, masked, 0, lim, sl2, neg_scale);
        float alpha = 1.f;
        bool upd = false;
        auto exps = [&]() {
          const float m_use = (m == -INFINITY) ? 0.f : m;
          const float2 negm = make_float2(-m_use, -m_use);
          float2 a4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                          make_float2(0.f, 0.f)};
          if (masked) {
#pragma unroll
            for (int k0 = 0; k0 < kBN; k0 += 16) {
              uint32_t pk[8];
              exp16<BF16, true>(sr, k0, c2, negm, 0, lim, a4, pk);
              tmem_st8(t_s + k0 / 2, pk);
            }
          } else {
#pragma unroll
            for (int k0 = 0; k0 < kBN; k0 += 16) {
              uint32_t pk[8];
              exp16<BF16, false>(sr, k0, c2, negm, 0, lim, a4, pk);
              tmem_st8(t_s + k0 / 2, pk);
            }
          }
          const float2 a = __fadd2_rn(__fadd2_rn(a4[0], a4[1]), __fadd2_rn(a4[2], a4[3]));
          return a.x + a.y;
        };
        float blk = exps();
        // Every P~ <= 2^8 holds if the block's sum does; otherwise (or on NaN)
        // move m to this block's maximum, rescale and redo the block.
        const bool need = !(blk <= kPSumLimit);
        if (__any_sync(0xffffffffu, need)) {
          const float m_blk = block_max_scaled<kBN>(sr, masked, 0, lim, sl2, neg_scale);
          if (need && m_blk > m) {
            alpha = ex2(m - m_blk);
            m = m_blk;
            upd = true;
          }
          if (__any_sync(0xffffffffu, upd)) {
            tmem_st_wait();  // the first pass's stores land before they are overwritten
            blk = exps();
            // O_t holds the blocks before j relative to the old m.
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
        warp_arrive(&bar_pfull[h]);
      }
      if (!alive) break;
      // ---------------------------------------------------------- epilogue
      if (!warp_wait(&bar_ofinal[h], on & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutSoftmax)) {
        alive = false;
        break;
      }
      ++on;
      tc_fence_after();
      const float inv_l = 1.f / l;
      const bool row_ok = row_g < S;
      const size_t o_row = static_cast<size_t>(bh) * S + (row_ok ? row_g : 0);
      elem_t* orow = reinterpret_cast<elem_t*>(p.o) + o_row * D;
#pragma unroll
      for (int c = 0; c < D; c += 16) {
        uint32_t o16[16];
        tmem_ld16(t_o + c, o16);
        if (row_ok) store_row16<BF16>(orow + c, o16, inv_l);
      }
      if (row_ok) p.lse[o_row] = (m + log2f(l)) * 0.69314718055994530942f;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kPMma0) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

namespace {
int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) ==
                                                  cudaSuccess)
      n = v;
    if (n <= 0) n = 1;
  }
  return n;
}

template <int D, bool BF16>
cudaError_t launch_fwd4p_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                           int BH, cudaStream_t stream) {
  using L = FPLayout<D>;
  auto kern = fa_fwd4p_kernel<D, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
  if (e != cudaSuccess) return e;
  // The register split assumes the launch gives exactly kPLaunchRegs per thread.
  cudaFuncAttributes attr;
  e = cudaFuncGetAttributes(&attr, kern);
  if (e != cudaSuccess) return e;
  if (attr.numRegs != kPLaunchRegs) return cudaErrorInvalidConfiguration;
  const int n_rb = (p.S + kPRowsPerItem - 1) / kPRowsPerItem;
  const int64_t n_items = static_cast<int64_t>(BH) * n_rb;
  if (n_items <= 0) return cudaSuccess;
  if (n_items > (1LL << 30)) return cudaErrorInvalidValue;
  const int64_t want = (n_items + kPPipes - 1) / kPPipes;
  const int grid = static_cast<int>(want < sm_count() ? want : sm_count());
  kern<<<grid, kPThreads, L::kSmemBytes, stream>>>(tq, tk, tv, p, static_cast<int>(n_items), n_rb);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_fwd4p(int D, bool bf16, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const FwdParams& p, int BH, cudaStream_t stream) {
  switch (D) {
    case 16:
      return bf16 ? launch_fwd4p_t<16, true>(tq, tk, tv, p, BH, stream)
                  : launch_fwd4p_t<16, false>(tq, tk, tv, p, BH, stream);
    case 32:
      return bf16 ? launch_fwd4p_t<32, true>(tq, tk, tv, p, BH, stream)
                  : launch_fwd4p_t<32, false>(tq, tk, tv, p, BH, stream);
    case 64:
      return bf16 ? launch_fwd4p_t<64, true>(tq, tk, tv, p, BH, stream)
                  : launch_fwd4p_t<64, false>(tq, tk, tv, p, BH, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace fa
