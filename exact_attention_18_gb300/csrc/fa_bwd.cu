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
//      over 64-row blocks of the queries that see it; dV and dK stay in TMEM;
//   3. bwd_main<KV_OUTER = false>: one CTA per (b*h, 128-query tile), looping
//      over 64-row blocks of its visible keys; dQ stays in TMEM.
// Causal: a key tile starts at its diagonal query block, a query tile stops at
// its diagonal key block (CS336 write-up, causal tile skipping); the mask is
// applied element-wise only on diagonal blocks and on ragged tails.
//
// bwd_main is written once for both passes.  Per partner block i it computes
// two score-shaped products with the CTA's resident 128-row tiles A1, A2 as
// the MMA A operands and the streamed 64-row tiles B1, B2 as B operands:
//   X = A1 B1^T,  Y = A2 B2^T
//     dK/dV pass: A1 = K, A2 = V, B1 = Q_i, B2 = dO_i -> X = S^T, Y = dP^T
//     dQ pass:    A1 = Q, A2 = dO, B1 = K_j, B2 = V_j -> X = S,   Y = dP
// so TMEM lane = the CTA's own row (key or query).  Sixteen softmax-gradient
// warps in two groups of eight turn X, Y into P and dS (16-bit, written back
// into TMEM over X and Y); group g takes the blocks i with i mod 2 = g, and in
// a group warp w owns TMEM lanes 32(w%4).. and partner columns 32((w/4)%2)...
// The MMA warp then accumulates, with A read from TMEM:
//     dK/dV pass: dV += P^T dO_i,  dK += dS^T Q_i    (B = B2, B1 read MN-major)
//     dQ pass:    dQ += dS K_j                       (B = B1 read MN-major)
// X and Y of block i live in TMEM buffer i mod kXYBufs (128 columns; three
// buffers for D <= 64, two for D = 128).  One warp issues X, Y of every block
// as soon as its tiles and buffer are free, another the accumulations, so a
// group that finishes block i usually finds block i + 2 already computed, and
// both groups work while the tensor core runs the products around them.  In the dK/dV pass the producer warp also copies the
// block's L and Delta (one value per partner query) into the stage with
// cp.async, completing on the same barrier as the block's tiles.
#include "fa_kernel_common.cuh"

namespace fa {
using namespace ptx;

// Source of L = +inf for partner query rows past a sample's end (dK/dV pass,
// general instantiation).
__device__ const float g_pos_inf = __builtin_huge_valf();

// ------------------------------------------------------------------ preprocess
// Delta_i = sum_d dO_id * O_id in fp32.  D/8 lanes share a row, each reading
// 16 bytes of O and of dO; a shuffle tree sums the group.  The whole warp
// calls it (the shuffles need all 32 lanes); `valid` says whether this lane's
// row exists.  Every lane of the group gets the row's sum.
// This lane's part of the row's dot product: 8 elements of O (a) and of dO (b).
template <bool BF16>
__device__ __forceinline__ float chunk_dot(const uint4 a, const uint4 b) {
  const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
  const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
  float acc = 0.f;
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
  return acc;
}

// Sum over the row's D/8 lanes.
template <int D>
__device__ __forceinline__ float row_sum(float acc) {
#pragma unroll
  for (int off = D / 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  return acc;
}

template <int D, bool BF16>
__device__ __forceinline__ float row_delta(const void* o, const void* dout, int64_t row, bool valid) {
  float acc = 0.f;
  if (valid) {
    const int64_t off = (row * D + ((threadIdx.x & 31) % (D / 8)) * 8) * 2;  // this lane's 8 elements
    acc = chunk_dot<BF16>(*reinterpret_cast<const uint4*>(static_cast<const char*>(o) + off),
                          *reinterpret_cast<const uint4*>(static_cast<const char*>(dout) + off));
  }
  return row_sum<D>(acc);
}

template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_preprocess_kernel(const BwdParams p, int64_t rows) {
  // The dK/dV pass after it may start its CTAs; it waits for this grid before reading Delta.
  griddep_launch_dependents();
  constexpr int kTpr = D / 8;           // threads per row
  constexpr int kRowsPerWarp = 32 / kTpr;
  const int lane = threadIdx.x & 31;
  const int sub = lane % kTpr;
  const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  // Whole warps iterate together so the shuffles always see 32 lanes.
  for (int64_t r0 = warp_id * kRowsPerWarp; r0 < rows; r0 += n_warps * kRowsPerWarp) {
    const int64_t row = r0 + lane / kTpr;
    const float acc = row_delta<D, BF16>(p.o, p.dout, row, row < rows);
    // Row `row` of [B*H*S, D] (fixed length) or of [T*H, D] (packed: token
    // row / H, head row % H, whose Delta lives at [head, token]).
    if (row < rows && sub == 0)
      p.delta[p.cu_seqlens ? (row % p.heads) * p.total + row / p.heads : row] = acc;
  }
}

// ------------------------------------------------------------------ dK/dV partial sums
// dV, dK = sum over the kv_splits partials (fixed order, fp32), rounded once.
// One thread per 8 consecutive columns of a [dV | scale*dK] row.
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_dkv_reduce_kernel(const BwdParams p, int64_t rows) {
  constexpr int kG = 2 * D / 8;  // 8-column groups per row
  const int64_t n = rows * kG;
  const int64_t part_stride = rows * 2 * D;
  for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = e / kG;
    const int cg = static_cast<int>(e - row * kG);
    const float* src = p.dkv_part + row * 2 * D + cg * 8;
    float4 a = reinterpret_cast<const float4*>(src)[0];
    float4 b = reinterpret_cast<const float4*>(src)[1];
    for (int sp = 1; sp < p.kv_splits; ++sp) {
      const float4 a2 = reinterpret_cast<const float4*>(src + sp * part_stride)[0];
      const float4 b2 = reinterpret_cast<const float4*>(src + sp * part_stride)[1];
      a.x += a2.x; a.y += a2.y; a.z += a2.z; a.w += a2.w;
      b.x += b2.x; b.y += b2.y; b.z += b2.z; b.w += b2.w;
    }
    const uint4 w = make_uint4(pack2<BF16>(a.x, a.y), pack2<BF16>(a.z, a.w), pack2<BF16>(b.x, b.y),
                               pack2<BF16>(b.z, b.w));
    const bool is_dv = cg < D / 8;
    void* out = is_dv ? p.dv : p.dk;
    const int col = (is_dv ? cg : cg - D / 8) * 8;
    reinterpret_cast<uint4*>(static_cast<char*>(out) + (row * D + col) * 2)[0] = w;
  }
}

namespace {

constexpr int kPartnerRows = 64;  // rows of a streamed B tile
constexpr int kBwdGroups = 2;     // softmax-gradient groups of 8 warps; group g takes blocks i = g mod 2
constexpr int kProducerWarp = 8 * kBwdGroups;
constexpr int kMmaWarp = kProducerWarp + 1;  // issues the score products X, Y
constexpr int kAccWarp = kMmaWarp + 1;       // issues the accumulations
constexpr int kBwdThreads = (kAccWarp + 1) * 32;
constexpr int kDeltaWarp = kAccWarp + 1;  // persistent dQ pass: computes Delta
constexpr int kDqpThreads = kBwdThreads + 32;
// "P and dS of block i stored" barriers, block i on bar_pfull[i % 4] (8
// arrivals, one per warp of group i % 2).  With three X/Y buffers a warp of a
// group may finish block i and move on to the group's next block, i + 2,
// before another warp of the group has finished block i: X, Y(i + 2) wait only
// for the accumulation of block i - 1, the other group's.  With one barrier
// per group the fast warp's next arrival would count toward block i's phase,
// which could then complete before all of block i's P and dS are stored; with
// two per group it lands on the other barrier.  No warp gets two blocks ahead:
// X, Y(i + 4) wait for an accumulation issued after block i's, which waits
// for all eight arrivals of block i.
constexpr int kPFullBars = 2 * kBwdGroups;

template <int D>
struct BwdLayout {
  using GA = TileGeom<D, 128>;
  using GB = TileGeom<D, kPartnerRows>;
  // Partner blocks in flight: enough to cover the load latency where shared
  // memory allows (D <= 64); D = 128 tiles leave room for four.
  static constexpr int kStages = D <= 64 ? 8 : 4;
  static constexpr int kOffA1 = 0;
  static constexpr int kOffA2 = kOffA1 + GA::kTileBytes;
  static constexpr int kOffB1 = kOffA2 + GA::kTileBytes;             // [kStages] tiles
  static constexpr int kOffB2 = kOffB1 + kStages * GB::kTileBytes;   // [kStages] tiles
  static constexpr int kOffVec = kOffB2 + kStages * GB::kTileBytes;  // [kStages][L, Delta][64] fp32
  static constexpr int kOffBar = kOffVec + kStages * 2 * kPartnerRows * 4;
  // X/Y buffers in TMEM (128 columns each): three when the accumulators
  // leave room (D <= 64), so the MMA warp can compute X, Y two blocks ahead.
  static constexpr int kXYBufs = D <= 64 ? 3 : 2;
  // a_full, b_full[S], empty[S], xy_full[buffers], acc_issued[buffers], p_full[4], acc_final, drain[2],
  // then (persistent kernels only) a_empty, acc_free, delta_full[2], delta_free[2], stage_full.
  static constexpr int kNumBars = 1 + 2 * kStages + 2 * kXYBufs + kPFullBars + 1 + 2 + 7;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemUsed = kOffMisc + 16;
  static constexpr int kSmemBytes = (kSmemUsed + 1024) > 116 * 1024 ? (kSmemUsed + 1024) : 116 * 1024;
  static constexpr uint32_t kTmemCols = 512;
  // Group g's buffer: X at column 128 g, Y at 128 g + 64 (64 fp32 columns each).
  static constexpr uint32_t kColAcc1 = 128 * kXYBufs;      // dV (dK/dV pass) or dQ
  static constexpr uint32_t kColAcc2 = 128 * kXYBufs + D;  // dK (dK/dV pass)
  static_assert(kColAcc2 + D <= kTmemCols, "TMEM layout");
  // dQ pass: the resident tiles A1 = Q, A2 = dO are copied into TMEM (D/2
  // columns each, after dQ; at D = 128 they take the columns dK would use in
  // the dK/dV pass) and the score products read A from there instead of
  // shared memory (32 instead of 48 cycles per M128 N64 K16 MMA).
  static constexpr bool kTmemA = true;
  static constexpr uint32_t kColA1 = kColAcc1 + D;
  static constexpr uint32_t kColA2 = kColA1 + D / 2;
  static_assert(!kTmemA || kColA2 + D / 2 <= kTmemCols, "TMEM layout");
};

// TMEM column (relative to a buffer's X or Y) of MMA K-step kk of the 16-bit
// P or dS block: warp half h wrote partner columns 32h..32h+31 packed into
// columns 32h..32h+15 of its own 32-column region.
__device__ __forceinline__ uint32_t packed_col(int kk) { return kk < 2 ? kk * 8 : 32 + (kk - 2) * 8; }


// One warp's 32 partner columns of a block: from the scores X and the
// gradient products Y (fp32, TMEM) form P = exp2(c X - L log2 e) and
// dS = P o (Y - Delta) and write them back as 16-bit pairs over the columns
// of X (P, dK/dV pass only) and Y (dS) already read.  In the dK/dV pass each
// column is a partner query whose L and Delta come from lv, dv; in the dQ
// pass they are the thread's own row's.  With DIAG the causal mask zeroes
// partner column c where c < lim (dK/dV pass) or c > lim (dQ pass); with WIN
// (a window band, dQ pass) also where c < lo.
template <bool BF16, bool KV_OUTER, bool DIAG, bool WIN = false>
__device__ __forceinline__ void grad_block(uint32_t tX, uint32_t tY, const float* lv, const float* dv, float2 c2,
                                           float my_l2, float my_delta, int lim, int lo = 0) {
  constexpr float kLog2e = 1.4426950408889634f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t xs[16], ys[16];
    tmem_ld16x2(tX + 16 * h, xs, tY + 16 * h, ys);
    uint32_t pk[8], dk[8];
#pragma unroll
    for (int c = 0; c < 16; c += 2) {
      const int cc = 16 * h + c;
      float2 nl2, dl;
      if constexpr (KV_OUTER) {
        nl2 = __fmul2_rn(make_float2(lv[cc], lv[cc + 1]), make_float2(-kLog2e, -kLog2e));
        dl = make_float2(dv[cc], dv[cc + 1]);
      } else {
        nl2 = make_float2(-my_l2, -my_l2);
        dl = make_float2(my_delta, my_delta);
      }
      const float2 y = __ffma2_rn(make_float2(__uint_as_float(xs[c]), __uint_as_float(xs[c + 1])), c2, nl2);
      float2 pr = make_float2(ex2(y.x), ex2(y.y));
      if constexpr (DIAG) {
        if ((KV_OUTER ? cc < lim : cc > lim) || (WIN && cc < lo)) pr.x = 0.f;
        if ((KV_OUTER ? cc + 1 < lim : cc + 1 > lim) || (WIN && cc + 1 < lo)) pr.y = 0.f;
      }
      const float2 gr = __fadd2_rn(make_float2(__uint_as_float(ys[c]), __uint_as_float(ys[c + 1])),
                                   make_float2(-dl.x, -dl.y));
      const float2 ds = __fmul2_rn(pr, gr);
      pk[c / 2] = pack2<BF16>(pr.x, pr.y);
      dk[c / 2] = pack2<BF16>(ds.x, ds.y);
    }
    // 16-bit P (dK/dV pass only) and dS of these 16 columns go to columns
    // 8h..8h+7 of this warp's region of X and Y, already read.
    if constexpr (KV_OUTER) tmem_st8(tX + 8 * h, pk);
    tmem_st8(tY + 8 * h, dk);
  }
}


// The dK/dV pass's version of grad_block, where the partner columns are
// queries with their own L and Delta.  The 32x32b layout would give every
// thread all 32 of the warp's columns and so all 32 (L, Delta) pairs from
// shared memory; with 16x256b loads a thread holds 2 adjacent columns of each
// of 4 column groups for 4 of the warp's rows (lanes t/4 + 8k), i.e. 8
// columns, a quarter of the shared-memory reads.  The packed 16-bit results
// of such a column pair go back with 16x128b stores to packed column
// (8i + 2(t%4)) / 2 = 4i + t%4, the layout the accumulation MMAs read.
// lim0: key index of the warp's first row minus its first partner column.
// With WIN (a window band) the mask keeps, for key row j, the partner
// queries j - wr .. j + wl: columns lim - wr .. lim + wl.
template <bool BF16, bool DIAG, bool WIN = false>
__device__ __forceinline__ void grad_block_kv(uint32_t tX, uint32_t tY, const float* lv, const float* dv, float2 c2,
                                              int lim0, int wr = 0, int wl = 0) {
  constexpr float kLog2e = 1.4426950408889634f;
  const int lane = threadIdx.x & 31;
  const int u = lane & 3;   // column pair within each group of 8
  const int r = lane >> 2;  // first of the thread's rows within 16
  float2 nl2[4], dl[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 l2 = *reinterpret_cast<const float2*>(lv + 8 * i + 2 * u);
    nl2[i] = __fmul2_rn(l2, make_float2(-kLog2e, -kLog2e));
    const float2 d2 = *reinterpret_cast<const float2*>(dv + 8 * i + 2 * u);
    dl[i] = make_float2(-d2.x, -d2.y);
  }
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const uint32_t lane_off = static_cast<uint32_t>(16 * half) << 16;
    uint32_t xs[16], ys[16];
    tmem_ld16x256b_x4(tX + lane_off, xs);
    tmem_ld16x256b_x4(tY + lane_off, ys);
    tmem_ld_wait();
    uint32_t pk[8], dk[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int e = 4 * i + 2 * k;
        const float2 y = __ffma2_rn(make_float2(__uint_as_float(xs[e]), __uint_as_float(xs[e + 1])), c2, nl2[i]);
        float2 pr = make_float2(ex2(y.x), ex2(y.y));
        if constexpr (DIAG) {
          const int lim = lim0 + 16 * half + r + 8 * k;  // zero partner columns c < lim (query before key)
          const int cc = 8 * i + 2 * u;
          if constexpr (WIN) {
            if (cc < lim - wr || cc > lim + wl) pr.x = 0.f;
            if (cc + 1 < lim - wr || cc + 1 > lim + wl) pr.y = 0.f;
          } else {
            if (cc < lim) pr.x = 0.f;
            if (cc + 1 < lim) pr.y = 0.f;
          }
        }
        const float2 gr = __fadd2_rn(make_float2(__uint_as_float(ys[e]), __uint_as_float(ys[e + 1])), dl[i]);
        const float2 ds = __fmul2_rn(pr, gr);
        pk[2 * i + k] = pack2<BF16>(pr.x, pr.y);
        dk[2 * i + k] = pack2<BF16>(ds.x, ds.y);
      }
    }
    tmem_st16x128b_x4(tX + lane_off, pk);
    tmem_st16x128b_x4(tY + lane_off, dk);
  }
}

}  // namespace

// GENERAL = true is the instantiation for packed variable-length batches and
// window bands (the layouts of BwdParams; "Inside FlashAttention" §6.1):
// the CTA finds its sample from cu_seqlens, streams only the partner blocks
// that meet its tile's band, and masks blocks crossing either band edge.
template <int D, bool BF16, bool KV_OUTER, bool GENERAL>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_main_kernel(const __grid_constant__ CUtensorMap tm_a1, const __grid_constant__ CUtensorMap tm_a2,
                       const __grid_constant__ CUtensorMap tm_b1, const __grid_constant__ CUtensorMap tm_b2,
                       const BwdParams p) {
  using L = BwdLayout<D>;
  using GA = typename L::GA;
  using GB = typename L::GB;
  using elem_t = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  constexpr int kPN = kPartnerRows;
  constexpr float kLog2e = 1.4426950408889634f;
  // Barrier tests before a wait blocks (mbar_wait): measured per pass at
  // causal B4 H16 S4096 D64 and B2 H32 S8192 D128 (a blocking try returns
  // some hundred cycles after the phase completes when the SM is busy): the
  // MMA warps gain in both passes except the D = 128 dQ pass, the other
  // waits only in the D <= 64 dK/dV pass; the dK/dV pass runs its tests
  // unrolled, the dQ pass eight per loop iteration.
  constexpr int kSpinMma = (D <= 64 || KV_OUTER) ? 64 : 0;
  constexpr int kSpinOther = (D <= 64 && KV_OUTER) ? 64 : 0;
  constexpr int kUnrollMma = (kSpinMma > 0 && KV_OUTER) ? kSpinMma : (kSpinMma > 0 ? 8 : 1);
  constexpr int kUnrollOther = kSpinOther > 0 ? kSpinOther : 1;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* bar_afull = bars;
  uint64_t* bar_bfull = bars + 1;
  uint64_t* bar_empty = bar_bfull + L::kStages;
  uint64_t* bar_xyfull = bar_empty + L::kStages;  // [buffers]
  uint64_t* bar_accissued = bar_xyfull + L::kXYBufs;  // [buffers] accumulation reading it issued
  uint64_t* bar_pfull = bar_accissued + L::kXYBufs;     // [4] block i's P, dS stored: bar_pfull[i % 4]
  uint64_t* bar_accfinal = bar_pfull + kPFullBars;
  uint64_t* bar_drain = bar_accfinal + 1;               // [2] one per MMA warp
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);
  float* vecs = reinterpret_cast<float*>(smem + L::kOffVec);

  const int warp = warp_index();
  const int lane = threadIdx.x & 31;
  // Head of the CTA's own tiles: a K/V head in the dK/dV pass, a query head in
  // the dQ pass.  K/V head h serves query heads h*group .. h*group+group-1; in
  // the dK/dV pass kv_splits CTAs share a K/V head, CTA `kv_part` taking the
  // group's heads kv_part*hpc .. kv_part*hpc+hpc-1.
  int cx, cy;
  cta_coords(!p.causal, &cx, &cy);
  const int bh = KV_OUTER ? cx / p.kv_splits : cx;
  const int kv_part = KV_OUTER ? cx - bh * p.kv_splits : 0;
  const int hpc = KV_OUTER ? p.group / p.kv_splits : 1;
  // General instantiation: the sample of a packed batch.  Head indices are
  // global (b*H + h) in the fixed-length layout and within a token when
  // packed: own_h for the CTA's own tiles, pz0 for the first partner head.
  const int heads_own = KV_OUTER ? p.heads / p.group : p.heads;  // per batch entry
  int S_ = p.S, tok0 = 0, own_h = bh;
  int pz0 = KV_OUTER ? bh * p.group + kv_part * hpc : bh / p.group;
  bool packed = false;
  if constexpr (GENERAL) {
    packed = p.cu_seqlens != nullptr;
    if (packed) {
      const int b = bh / heads_own;
      if (!packed_sample(p.cu_seqlens, b, p.S, p.total, p.err, &tok0, &S_)) return;
      own_h = bh - b * heads_own;
      pz0 = KV_OUTER ? own_h * p.group + kv_part * hpc : own_h / p.group;
    }
  }
  const int S = S_;
  const int nt = p.n_tiles;
  const int np = (S + kPN - 1) / kPN;
  const int64_t rowbase = static_cast<int64_t>(bh) * S;
  // Row r of head h: L and Delta at h * lstride + loff + r (general instantiation).
  const int lstride = (GENERAL && packed) ? p.total : S;
  const int loff = tok0;
  // Own tile; heavy tiles first under the causal mask (key tile 0 and query
  // tile nt-1 see the most partners).
  const int own = KV_OUTER ? cy : (p.causal ? nt - 1 - cy : cy);
  const int own0 = own * 128;
  if constexpr (GENERAL) {
    if (own0 >= S) return;  // packed batch: this CTA lies past its sample
  }
  // Window (general instantiation): key j is visible to query i iff i - wl <= j <= i + wr.
  const int wl = GENERAL ? p.win_left : 0;
  const int wr = GENERAL ? p.win_right : 0;
  // Partner blocks [first, last_excl): queries j - wr .. j + wl of the tile's
  // keys (dK/dV pass) or keys i - wl .. i + wr of its queries (dQ pass).
  int first, last_excl;
  if constexpr (GENERAL) {
    const int below = KV_OUTER ? wr : wl, above = KV_OUTER ? wl : wr;
    first = max(0, own0 - below) / kPN;
    last_excl = min(np, min(S - 1, own0 + 127 + above) / kPN + 1);
  } else {
    first = (KV_OUTER && p.causal) ? own0 / kPN : 0;
    last_excl = (!KV_OUTER && p.causal) ? min(np, (own0 + 127) / kPN + 1) : np;
  }
  // Partner blocks per partner head; the dK/dV pass streams them for each of
  // the group's query heads in turn and sums over all of them.
  const int nper = last_excl - first;
  const int niter = KV_OUTER ? hpc * nper : nper;

  if (threadIdx.x == 0) {
    mbar_init(bar_afull, 1);
    for (int s = 0; s < L::kStages; ++s) {
      // dK/dV pass: the producer's TMA arrival plus one cp.async arrival per
      // producer lane for the block's L and Delta vectors.
      mbar_init(&bar_bfull[s], KV_OUTER ? 33 : 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int b = 0; b < L::kXYBufs; ++b) {
      mbar_init(&bar_xyfull[b], 1);
      mbar_init(&bar_accissued[b], 1);
    }
    for (int b = 0; b < kPFullBars; ++b) {
      mbar_init(&bar_pfull[b], 8);  // one arrival per warp of the block's group
    }
    mbar_init(bar_accfinal, 1);
    mbar_init(&bar_drain[0], 1);
    mbar_init(&bar_drain[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
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
  // The dQ pass after the dK/dV pass may start its CTAs as this grid's last
  // ones run; it reads nothing this pass writes before its griddep_wait.
  if constexpr (KV_OUTER) griddep_launch_dependents();

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    // Lane 0 issues the TMA copies; in the dK/dV pass every lane also copies
    // two entries of the block's L and Delta vectors (queries past S read 0:
    // their Q and dO rows are zero-filled, so P dO and dS vanish there).
    if (lane == 0) {
      prefetch_tmap(&tm_a1);
      prefetch_tmap(&tm_a2);
      prefetch_tmap(&tm_b1);
      prefetch_tmap(&tm_b2);
      mbar_arrive_expect_tx(bar_afull, 2 * GA::kTileBytes);
#pragma unroll
      for (int ch = 0; ch < GA::kChunks; ++ch) {
        tma_load_3d(smem + L::kOffA1 + ch * GA::kChunkBytes, &tm_a1, bar_afull, ch * (GA::kRowBytes / 2),
                    (GENERAL && packed) ? own_h : own0, (GENERAL && packed) ? tok0 + own0 : own_h);
        tma_load_3d(smem + L::kOffA2 + ch * GA::kChunkBytes, &tm_a2, bar_afull, ch * (GA::kRowBytes / 2),
                    (GENERAL && packed) ? own_h : own0, (GENERAL && packed) ? tok0 + own0 : own_h);
      }
    }
    int it = 0;
    // Partner head and block of iteration `it`, stepped along without divisions.
    int pz = pz0;
    int pblk = first;
    for (; it < niter; ++it, ++pblk) {
      if (KV_OUTER && pblk == last_excl) {
        pblk = first;
        ++pz;
      }
      const int st = it % L::kStages;
      const int use = it / L::kStages;
      if (use > 0 && !warp_wait<kSpinOther, kUnrollOther>(&bar_empty[st], (use - 1) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutLoad)) break;
      const int r0 = pblk * kPN;
      if (lane == 0) {
        mbar_arrive_expect_tx(&bar_bfull[st], 2 * GB::kTileBytes);
#pragma unroll
        for (int ch = 0; ch < GB::kChunks; ++ch) {
          tma_load_3d(smem + L::kOffB1 + st * GB::kTileBytes + ch * GB::kChunkBytes, &tm_b1, &bar_bfull[st],
                      ch * (GB::kRowBytes / 2), (GENERAL && packed) ? pz : r0, (GENERAL && packed) ? tok0 + r0 : pz);
          tma_load_3d(smem + L::kOffB2 + st * GB::kTileBytes + ch * GB::kChunkBytes, &tm_b2, &bar_bfull[st],
                      ch * (GB::kRowBytes / 2), (GENERAL && packed) ? pz : r0, (GENERAL && packed) ? tok0 + r0 : pz);
        }
      }
      if constexpr (KV_OUTER) {
        // Delta may come from the kernel just before this one (a programmatic
        // dependent launch after the persistent dQ pass): wait for it before the
        // first read.  Nothing read earlier is written by that kernel.
        if (it == 0) griddep_wait();
        float* v = vecs + st * 2 * kPN;
#pragma unroll
        for (int h = 0; h < kPN; h += 32) {
          const int q = r0 + h + lane;
          if constexpr (GENERAL) {
            // Partner queries past the sample read L = +inf and Delta = 0, so
            // their P and dS are exactly 0 (when packed, their Q and dO rows
            // are the next sample's).
            const int64_t src = static_cast<int64_t>(pz) * lstride + loff + (q < S ? q : S - 1);
            cp_async_4(v + h + lane, q < S ? p.lse + src : &g_pos_inf, true);
            cp_async_4(v + kPN + h + lane, p.delta + src, q < S);
          } else {
            const int64_t src = static_cast<int64_t>(pz) * S + (q < S ? q : S - 1);
            cp_async_4(v + h + lane, p.lse + src, q < S);
            cp_async_4(v + kPN + h + lane, p.delta + src, q < S);
          }
        }
        cp_async_mbar_arrive(&bar_bfull[st]);
      }
    }
    // A CTA with no partner block (a key tile past a short sample's end) still
    // waits for the kernel before it, so that this grid never completes before
    // that one, whatever follows on the stream.
    if constexpr (KV_OUTER) {
      if (it == 0) griddep_wait();
    }
    // Teardown: every copy issued must land before the CTA exits.
    if (lane == 0) drain_wait(bar_afull, 0, p.err);
    for (int x = (it > L::kStages ? it - L::kStages : 0); x < it; ++x)
      drain_wait(&bar_bfull[x % L::kStages], (x / L::kStages) & 1, p.err);
  } else if (warp == kMmaWarp || warp == kAccWarp) {
    // ------------------------------------------------------------ MMA issuers
    // Warp kMmaWarp issues the score products X, Y of every block, warp
    // kAccWarp the accumulations, so X, Y keep the tensor core busy while the
    // accumulation of a block waits for its P and dS.  Both run converged and
    // one elected lane issues each MMA.  X, Y(i) reuse buffer i % kXYBufs,
    // last read by the accumulation of block i - kXYBufs: kAccWarp signals
    // acc_issued after issuing it (tcgen05 fences order the two warps' MMAs,
    // which the tensor core then runs in issue order).
    constexpr uint32_t idesc_xy = make_idesc_f16(BF16, 128, kPN, false, false);
    constexpr uint32_t idesc_acc = make_idesc_f16(BF16, 128, D, false, true);
    const AccFlags accf = runtime_flags(S);
    bool ok = true;
    if (warp == kMmaWarp) {
      const uint64_t a1_desc = make_sdesc(sA1, 16, 8 * GA::kRowBytes, GA::kSwz);
      const uint64_t a2_desc = make_sdesc(sA2, 16, 8 * GA::kRowBytes, GA::kSwz);
      ok = warp_wait(bar_afull, 0, abort_flag, p.err, p.wait_ns, kErrTimeoutMma);
      constexpr bool kAFromTmem = !KV_OUTER && L::kTmemA;
      if (kAFromTmem && ok) {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          tmem_cp_128x256b_warp(tmem + L::kColA1 + 8 * kk, desc_plus(a1_desc, kmajor_step_bytes<D, 128>(kk)));
          tmem_cp_128x256b_warp(tmem + L::kColA2 + 8 * kk, desc_plus(a2_desc, kmajor_step_bytes<D, 128>(kk)));
        }
      }
      for (int i = 0; ok && i < niter; ++i) {
        const int st = i % L::kStages;
        const int b = i % L::kXYBufs;
        ok = warp_wait<kSpinMma, kUnrollMma>(&bar_bfull[st], (i / L::kStages) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutMma);
        if (ok && i >= L::kXYBufs)
          ok = warp_wait<kSpinMma, kUnrollMma>(&bar_accissued[b], ((i / L::kXYBufs) - 1) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutMma);
        if (!ok) break;
        tc_fence_after();
        const uint32_t tb = tmem + 128u * b;
        const uint64_t b1 = make_sdesc(sB1 + st * GB::kTileBytes, 16, 8 * GB::kRowBytes, GB::kSwz);
        const uint64_t b2 = make_sdesc(sB2 + st * GB::kTileBytes, 16, 8 * GB::kRowBytes, GB::kSwz);
        if constexpr (kAFromTmem) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ts_warp(tb, tmem + L::kColA1 + 8 * kk, desc_plus(b1, kmajor_step_bytes<D, kPN>(kk)), idesc_xy,
                        kk > 0 ? accf.on : accf.off);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ts_warp(tb + 64, tmem + L::kColA2 + 8 * kk, desc_plus(b2, kmajor_step_bytes<D, kPN>(kk)), idesc_xy,
                        kk > 0 ? accf.on : accf.off);
        } else {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss_warp(tb, desc_plus(a1_desc, kmajor_step_bytes<D, 128>(kk)),
                        desc_plus(b1, kmajor_step_bytes<D, kPN>(kk)), idesc_xy, kk > 0 ? accf.on : accf.off);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss_warp(tb + 64, desc_plus(a2_desc, kmajor_step_bytes<D, 128>(kk)),
                        desc_plus(b2, kmajor_step_bytes<D, kPN>(kk)), idesc_xy, kk > 0 ? accf.on : accf.off);
        }
        mma_commit_warp(&bar_xyfull[b]);
      }
      mma_commit_warp(&bar_drain[0]);
      drain_wait(&bar_drain[0], 0, p.err);
    } else {
      for (int x = 0; ok && x < niter; ++x) {
        const int st = x % L::kStages;
        const int b = x % L::kXYBufs;
        ok = warp_wait<kSpinMma, kUnrollMma>(&bar_pfull[x % kPFullBars], (x / kPFullBars) & 1, abort_flag, p.err, p.wait_ns,
                                             kErrTimeoutMma);
        if (!ok) break;
        tc_fence_after();
        const uint32_t tb = tmem + 128u * b;
        const uint64_t b1 = make_sdesc(sB1 + st * GB::kTileBytes, GB::kChunkBytes, 8 * GB::kRowBytes, GB::kSwz);
        const uint64_t b2 = make_sdesc(sB2 + st * GB::kTileBytes, GB::kChunkBytes, 8 * GB::kRowBytes, GB::kSwz);
        if constexpr (KV_OUTER) {
#pragma unroll
          for (int kk = 0; kk < kPN / 16; ++kk)  // dV += P^T dO_i
            mma_ts_warp(tmem + L::kColAcc1, tb + packed_col(kk), desc_plus(b2, mnmajor_step_bytes<D>(kk)), idesc_acc,
                        (x > 0 || kk > 0) ? accf.on : accf.off);
#pragma unroll
          for (int kk = 0; kk < kPN / 16; ++kk)  // dK += dS^T Q_i
            mma_ts_warp(tmem + L::kColAcc2, tb + 64 + packed_col(kk), desc_plus(b1, mnmajor_step_bytes<D>(kk)),
                        idesc_acc, (x > 0 || kk > 0) ? accf.on : accf.off);
        } else {
#pragma unroll
          for (int kk = 0; kk < kPN / 16; ++kk)  // dQ += dS K_j
            mma_ts_warp(tmem + L::kColAcc1, tb + 64 + packed_col(kk), desc_plus(b1, mnmajor_step_bytes<D>(kk)),
                        idesc_acc, (x > 0 || kk > 0) ? accf.on : accf.off);
        }
        // The stage's tiles are free once this completes: X, Y(x) finished
        // before the group could form P and dS.
        mma_commit_warp(&bar_empty[st]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_accissued[b]);
      }
      if (ok) mma_commit_warp(bar_accfinal);
      mma_commit_warp(&bar_drain[1]);
      drain_wait(&bar_drain[1], 0, p.err);
    }
  } else {
    // ------------------------------------------------------------ softmax-gradient warps 0-15
    // Group g = warp / 8 turns blocks g, g + 2, ... into P and dS, so two
    // blocks are in this stage at once while the tensor core works on a
    // third.  In a group, warp w owns TMEM lanes 32 (w % 4).. and partner
    // columns 32 ((w / 4) % 2)...
    const int g = warp >> 3;
    const int q4 = warp & 3;
    const int hf = (warp >> 2) & 1;
    const int col0 = 32 * hf;
    const int my = own0 + q4 * 32 + lane;  // key index (dK/dV pass) or query index (dQ pass)
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    const float sl2 = p.scale_log2;
    const float2 c2 = make_float2(sl2, sl2);
    // dQ pass: this thread's query row owns its L2 = L * log2 e and Delta
    // (rows past S: L2 = +inf, so their probabilities are exactly 0).
    float my_l2 = INFINITY, my_delta = 0.f;
    // Delta comes from a kernel before this one, which may still be running
    // when this pass is a programmatic dependent launch.
    if (!KV_OUTER) griddep_wait();
    if (!KV_OUTER && my < S) {
      const int64_t li = GENERAL ? static_cast<int64_t>(own_h) * lstride + loff + my : rowbase + my;
      my_l2 = p.lse[li] * kLog2e;
      my_delta = p.delta[li];
    }
    bool alive = true;
    int pi = g;  // i modulo nper: the partner block within its head (dK/dV pass)
    if constexpr (KV_OUTER) {
      while (pi >= nper) pi -= nper;
    }
    for (int i = g; i < niter; i += kBwdGroups) {
      const int st = i % L::kStages;
      const int partner0 = (first + (KV_OUTER ? pi : i)) * kPN;
      if constexpr (KV_OUTER) {
        pi += kBwdGroups;
        while (pi >= nper) pi -= nper;
      }
      bool ok = true;
      if constexpr (KV_OUTER) ok = warp_wait<kSpinOther, kUnrollOther>(&bar_bfull[st], (i / L::kStages) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutSoftmax);
      ok = ok && warp_wait<kSpinOther, kUnrollOther>(&bar_xyfull[i % L::kXYBufs], (i / L::kXYBufs) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutSoftmax);
      if (!ok) {
        alive = false;
        break;
      }
      tc_fence_after();
      const uint32_t tX = tmem + lane_base + 128u * (i % L::kXYBufs) + col0;
      const uint32_t tY = tX + 64;
      const float* lv = vecs + st * 2 * kPN + col0;  // L of this warp's 32 partner queries (dK/dV pass)
      const float* dv = lv + kPN;                    // and their Delta
      // Diagonal blocks under the causal mask: the dK/dV pass zeroes partner
      // column c where query partner0 + col0 + c < key `my`, the dQ pass where
      // key partner0 + col0 + c > query `my`.  Rows and columns past S need no
      // mask: their zero-filled operands make their terms vanish (see above).
      // Off-diagonal blocks (all but one or two per tile) take the path with
      // no per-element compare or select.
      if constexpr (GENERAL) {
        // Window band: blocks crossing either edge are masked; the dQ pass
        // also masks a packed sample's ragged last key block (those rows are
        // the next sample's).  Partner queries past S have P = 0 from L = +inf.
        if constexpr (KV_OUTER) {
          const bool edge = partner0 < own0 + 127 - wr || partner0 + kPN - 1 > own0 + wl;
          const int lim0 = own0 + q4 * 32 - partner0 - col0;
          if (edge)
            grad_block_kv<BF16, true, true>(tX, tY, lv, dv, c2, lim0, wr, wl);
          else
            grad_block_kv<BF16, false>(tX, tY, lv, dv, c2, lim0);
        } else {
          const bool edge = partner0 + kPN - 1 > own0 + wr || partner0 < own0 + 127 - wl ||
                            (packed && partner0 + kPN > S);
          const int hi = min(S - 1, my + wr) - partner0 - col0;
          const int lo = my - wl - partner0 - col0;
          if (edge)
            grad_block<BF16, KV_OUTER, true, true>(tX, tY, lv, dv, c2, my_l2, my_delta, hi, lo);
          else
            grad_block<BF16, KV_OUTER, false>(tX, tY, lv, dv, c2, my_l2, my_delta, hi);
        }
      } else {
        const bool diag = p.causal && (KV_OUTER ? partner0 < own0 + 128 : partner0 + kPN - 1 > own0);
        const int lim = my - partner0 - col0;
        if constexpr (KV_OUTER) {
          const int lim0 = own0 + q4 * 32 - partner0 - col0;
          if (diag)
            grad_block_kv<BF16, true>(tX, tY, lv, dv, c2, lim0);
          else
            grad_block_kv<BF16, false>(tX, tY, lv, dv, c2, lim0);
        } else {
          if (diag)
            grad_block<BF16, KV_OUTER, true>(tX, tY, lv, dv, c2, my_l2, my_delta, lim);
          else
            grad_block<BF16, KV_OUTER, false>(tX, tY, lv, dv, c2, my_l2, my_delta, lim);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_pfull[i % kPFullBars]);
    }
    // ------------------------------------------------------------ epilogue
    const bool done = alive && mbar_wait<kSpinOther, kUnrollOther>(bar_accfinal, 0, abort_flag, p.err, p.wait_ns, kErrTimeoutSoftmax);
    // The 16 warps split the accumulator columns of their 32 rows into up to
    // four parts of at least 16 columns.
    constexpr int kParts = D >= 64 ? 4 : D / 16;
    constexpr int kEpiCols = D / kParts;
    const int col_part = warp >> 2;
    if (__all_sync(0xffffffffu, done) && col_part < kParts) {
      tc_fence_after();
      const int c_begin = col_part * kEpiCols;
      const bool row_ok = my < S;
      // Output row: bh*S + my (fixed length) or (tok0 + my)*heads_own + own_h (packed).
      const int mr = row_ok ? my : 0;
      const int64_t orow = (GENERAL && packed) ? static_cast<int64_t>(tok0 + mr) * heads_own + own_h : rowbase + mr;
      const size_t off = static_cast<size_t>(orow) * D;
      const uint32_t t_acc = tmem + lane_base;
      if constexpr (KV_OUTER) {
        if (p.kv_splits == 1) {
          elem_t* dv_row = reinterpret_cast<elem_t*>(p.dv) + off;
          elem_t* dk_row = reinterpret_cast<elem_t*>(p.dk) + off;
#pragma unroll
          for (int c = c_begin; c < c_begin + kEpiCols; c += 16) {
            uint32_t v16[16];
            tmem_ld16(t_acc + L::kColAcc1 + c, v16);
            if (row_ok) store_row16<BF16>(dv_row + c, v16, 1.f);
            tmem_ld16(t_acc + L::kColAcc2 + c, v16);
            if (row_ok) store_row16<BF16>(dk_row + c, v16, p.scale);
          }
        } else {
          // This CTA's share of the group: fp32 rows [dV | scale * dK] of
          // partial `kv_part`, summed by the reduce kernel.
          const int64_t n_rows = (GENERAL && packed) ? static_cast<int64_t>(p.total) * heads_own
                                                     : static_cast<int64_t>(p.BH / p.group) * S;
          float* prow = p.dkv_part + ((static_cast<int64_t>(kv_part) * n_rows + orow) * (2 * D));
#pragma unroll
          for (int c = c_begin; c < c_begin + kEpiCols; c += 16) {
            uint32_t v16[16];
            tmem_ld16(t_acc + L::kColAcc1 + c, v16);
            if (row_ok) store_row16_f32(prow + c, v16, 1.f);
            tmem_ld16(t_acc + L::kColAcc2 + c, v16);
            if (row_ok) store_row16_f32(prow + D + c, v16, p.scale);
          }
        }
      } else {
        elem_t* dq_row = reinterpret_cast<elem_t*>(p.dq) + off;
#pragma unroll
        for (int c = c_begin; c < c_begin + kEpiCols; c += 16) {
          uint32_t v16[16];
          tmem_ld16(t_acc + L::kColAcc1 + c, v16);
          if (row_ok) store_row16<BF16>(dq_row + c, v16, p.scale);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}


// Persistent version of the dQ pass for fixed-length calls at D <= 64: a grid
// of at most one CTA per SM, each running the pipeline of fa_bwd_main_kernel
// (roles, TMEM layout, barriers; Q and dO copied into TMEM) over a sequence of
// the non-persistent grid's query tiles ("work items", in that grid's launch
// order: heaviest first under the causal mask), dealt to the CTAs in a snake
// (round r gives item r*P + c to CTA c when r is even and r*P + P-1-c when it
// is odd, P CTAs).  Between items nothing drains: the producer loads the next
// item's first key blocks, then its Q and dO tiles as soon as the current
// item's copies of them into TMEM are done (a_empty); the score-product warp
// computes the next item's first X, Y while the softmax-gradient warps store
// the current item's dQ; the accumulation warp starts the next item's dQ once
// those stores have read it out of TMEM (acc_free).  Barrier phases run on
// across items: key stages, X/Y buffers and the "P stored" barriers by a
// running block count, the tile and accumulator barriers by item.
// One more warp computes Delta = rowsum(dO o O) of each item's rows (the
// preprocess kernel's arithmetic, from O and dO rows staged in shared memory
// one item ahead), writes it to the workspace for the dK/dV pass, which then
// runs after this one, and hands it to the softmax-gradient warps through
// shared memory (delta_full), so the backward needs no separate Delta kernel.
template <int D>
struct DqpLayout {
  static constexpr int kOffStage = (BwdLayout<D>::kSmemUsed + 127) / 128 * 128;
  static constexpr int kStageBytes = 128 * D * 2;  // one item's rows of one tensor
  static constexpr int kSmemBytes = kOffStage + 2 * kStageBytes + 1024;
  static_assert(kSmemBytes <= 227 * 1024, "persistent dQ pass: shared memory");
};

template <int D, bool BF16>
__global__ void __launch_bounds__(kDqpThreads, 1)
    fa_bwd_dqp_kernel(const __grid_constant__ CUtensorMap tm_a1, const __grid_constant__ CUtensorMap tm_a2,
                      const __grid_constant__ CUtensorMap tm_b1, const __grid_constant__ CUtensorMap tm_b2,
                      const BwdParams p, int n_items) {
  using L = BwdLayout<D>;
  using DL = DqpLayout<D>;
  static_assert(D <= 64 && L::kTmemA, "persistent dQ pass: D <= 64, Q and dO in TMEM");
  using GA = typename L::GA;
  using GB = typename L::GB;
  using elem_t = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  constexpr int kPN = kPartnerRows;
  constexpr float kLog2e = 1.4426950408889634f;
  constexpr int kS = L::kStages;
  constexpr int kB = L::kXYBufs;
  // Barrier tests before blocking as in fa_bwd_main_kernel's dQ pass at D <= 64.
  constexpr int kSpinMma = 64;
  constexpr int kUnrollMma = 8;
  constexpr int kPreBlocks = 4;  // key blocks of the next item loaded before its Q, dO tiles

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* bar_afull = bars;
  uint64_t* bar_bfull = bars + 1;
  uint64_t* bar_empty = bar_bfull + kS;
  uint64_t* bar_xyfull = bar_empty + kS;         // [buffers]
  uint64_t* bar_accissued = bar_xyfull + kB;     // [buffers] accumulation reading it issued
  uint64_t* bar_pfull = bar_accissued + kB;      // [4] block i's dS stored: bar_pfull[i % 4]
  uint64_t* bar_accfinal = bar_pfull + kPFullBars;
  uint64_t* bar_drain = bar_accfinal + 1;        // [2] one per MMA warp
  uint64_t* bar_aempty = bar_drain + 2;          // the item's Q, dO copies into TMEM done
  uint64_t* bar_accfree = bar_aempty + 1;        // the item's dQ read out by all 16 warps
  uint64_t* bar_deltafull = bar_accfree + 1;     // [2] item n's Delta in buffer n % 2
  uint64_t* bar_deltafree = bar_deltafull + 2;   // [2] buffer n % 2 read by all 16 warps
  uint64_t* bar_stage = bar_deltafree + 2;       // an item's O, dO rows in the staging buffer
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);
  // Two 128-row Delta buffers (item n in buffer n % 2), in the stage vectors'
  // space, which the dQ pass does not use.
  float* delta_buf = reinterpret_cast<float*>(smem + L::kOffVec);
  static_assert(L::kStages * 2 * kPartnerRows >= 2 * 128, "Delta buffers");

  const int warp = warp_index();
  const int lane = threadIdx.x & 31;
  const int S = p.S;
  const int nt = p.n_tiles;
  const int np = (S + kPN - 1) / kPN;
  const int gx = p.BH;
  const int P = static_cast<int>(gridDim.x);
  const int c = static_cast<int>(blockIdx.x);
  auto item_at = [&](int r) -> int {
    const int k = r * P + ((r & 1) ? (P - 1 - c) : c);
    return k < n_items ? k : -1;
  };
  // One work item: query head bh, its 128-row tile at own0, key blocks 0 .. nb-1.
  struct Item {
    int bh, kvh, own0, nb;
  };
  auto decode = [&](int k) -> Item {
    int cx, cy;
    if (p.causal) {  // x fastest: every head's heaviest tile first
      cy = k / gx;
      cx = k - cy * gx;
    } else {         // y fastest: one head's tiles in a row
      cx = k / nt;
      cy = k - cx * nt;
    }
    Item it;
    it.bh = cx;
    it.kvh = cx / p.group;
    it.own0 = (p.causal ? nt - 1 - cy : cy) * 128;
    it.nb = p.causal ? min(np, (it.own0 + 127) / kPN + 1) : np;
    return it;
  };

  if (threadIdx.x == 0) {
    mbar_init(bar_afull, 1);
    for (int s = 0; s < kS; ++s) {
      mbar_init(&bar_bfull[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int b = 0; b < kB; ++b) {
      mbar_init(&bar_xyfull[b], 1);
      mbar_init(&bar_accissued[b], 1);
    }
    for (int b = 0; b < kPFullBars; ++b) mbar_init(&bar_pfull[b], 8);
    mbar_init(bar_accfinal, 1);
    mbar_init(&bar_drain[0], 1);
    mbar_init(&bar_drain[1], 1);
    mbar_init(bar_aempty, 1);
    mbar_init(bar_accfree, 16);  // one arrival per softmax-gradient warp
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bar_deltafull[b], 1);
      mbar_init(&bar_deltafree[b], 16);  // one arrival per softmax-gradient warp
    }
    mbar_init(bar_stage, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
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
  // The dK/dV pass that follows may start its CTAs as this grid's CTAs exit
  // (it cannot share an SM with one: registers); it waits for this grid to
  // complete before it reads Delta.
  griddep_launch_dependents();

  if (warp == kDeltaWarp) {
    // ------------------------------------------------------------ Delta warp
    // Lane 0 copies an item's O and dO rows into the staging buffer (one bulk
    // copy each: a fixed-length head's rows are contiguous), one item ahead of
    // the sums; D/8 lanes per row then sum dO o O from shared memory.
    constexpr int kTpr = D / 8;
    constexpr int kRowsPerStep = 32 / kTpr;
    uint8_t* stage_o = smem + DL::kOffStage;
    uint8_t* stage_do = stage_o + DL::kStageBytes;
    auto issue = [&](const Item& w) {
      const uint32_t bytes = static_cast<uint32_t>(min(128, S - w.own0)) * D * 2;
      const int64_t off = (static_cast<int64_t>(w.bh) * S + w.own0) * D * 2;
      mbar_arrive_expect_tx(bar_stage, 2 * bytes);
      // Evict-first: these lines are not read again soon (the item's dO tile
      // comes in through its own TMA load), and K, V blocks keep their L2 place.
      const uint64_t pol = l2_policy_evict_first();
      bulk_load(stage_o, static_cast<const char*>(p.o) + off, bytes, bar_stage, pol);
      bulk_load(stage_do, static_cast<const char*>(p.dout) + off, bytes, bar_stage, pol);
    };
    bool ok = true;
    int k = item_at(0);
    if (k >= 0 && lane == 0) issue(decode(k));
    int n = 0;  // item n's copy is the one in flight
    for (int r = 0; ok && k >= 0; ++r, ++n) {
      const Item w = decode(k);
      const int64_t rowbase = static_cast<int64_t>(w.bh) * S;
      // Buffer n % 2 was last read at the start of item n - 2.
      if (n >= 2)
        ok = warp_wait(&bar_deltafree[n & 1], ((n >> 1) - 1) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutSoftmax);
      if (ok) ok = warp_wait(bar_stage, n & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutSoftmax);
      if (!ok) break;
      float* buf = delta_buf + (n & 1) * 128;
      const int sub16 = (lane % kTpr) * 16;
#pragma unroll 4
      for (int r0 = 0; r0 < 128; r0 += kRowsPerStep) {
        const int rr = r0 + lane / kTpr;
        const int row = w.own0 + rr;
        float acc = 0.f;
        if (row < S)
          acc = chunk_dot<BF16>(*reinterpret_cast<const uint4*>(stage_o + rr * D * 2 + sub16),
                                *reinterpret_cast<const uint4*>(stage_do + rr * D * 2 + sub16));
        const float d = row_sum<D>(acc);
        if (lane % kTpr == 0) {
          buf[rr] = d;
          if (row < S) p.delta[rowbase + row] = d;
        }
      }
      k = item_at(r + 1);
      __syncwarp();
      if (lane == 0) {
        if (k >= 0) {  // the staging buffer is free again: the next item's rows
          fence_proxy_async_smem();
          issue(decode(k));
        }
        mbar_arrive(&bar_deltafull[n & 1]);  // release: the buffer's writes reach its waiters
      }
    }
    // Given up: the copy in flight lands before the CTA exits.
    if (!ok && lane == 0) drain_wait(bar_stage, n & 1, p.err);
  } else if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer (lane 0)
    if (lane == 0) {
      prefetch_tmap(&tm_a1);
      prefetch_tmap(&tm_a2);
      prefetch_tmap(&tm_b1);
      prefetch_tmap(&tm_b2);
      bool ok = true;
      int it = 0;  // key blocks loaded so far
      int n = 0;   // items whose Q, dO tiles were loaded
      for (int r = 0; ok; ++r) {
        const int k = item_at(r);
        if (k < 0) break;
        const Item w = decode(k);
        auto load_block = [&](int x) -> bool {
          const int st = it % kS;
          const int use = it / kS;
          if (use > 0 && !mbar_wait(&bar_empty[st], (use - 1) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutLoad))
            return false;
          mbar_arrive_expect_tx(&bar_bfull[st], 2 * GB::kTileBytes);
#pragma unroll
          for (int ch = 0; ch < GB::kChunks; ++ch) {
            tma_load_3d(smem + L::kOffB1 + st * GB::kTileBytes + ch * GB::kChunkBytes, &tm_b1, &bar_bfull[st],
                        ch * (GB::kRowBytes / 2), x * kPN, w.kvh);
            tma_load_3d(smem + L::kOffB2 + st * GB::kTileBytes + ch * GB::kChunkBytes, &tm_b2, &bar_bfull[st],
                        ch * (GB::kRowBytes / 2), x * kPN, w.kvh);
          }
          ++it;
          return true;
        };
        const int pre = min(w.nb, kPreBlocks);
        for (int x = 0; ok && x < pre; ++x) ok = load_block(x);
        // Q and dO, once the previous item's copies of them into TMEM are done.
        if (ok && n > 0) ok = mbar_wait(bar_aempty, (n - 1) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutLoad);
        if (!ok) break;
        mbar_arrive_expect_tx(bar_afull, 2 * GA::kTileBytes);
#pragma unroll
        for (int ch = 0; ch < GA::kChunks; ++ch) {
          tma_load_3d(smem + L::kOffA1 + ch * GA::kChunkBytes, &tm_a1, bar_afull, ch * (GA::kRowBytes / 2), w.own0,
                      w.bh);
          tma_load_3d(smem + L::kOffA2 + ch * GA::kChunkBytes, &tm_a2, bar_afull, ch * (GA::kRowBytes / 2), w.own0,
                      w.bh);
        }
        ++n;
        for (int x = pre; ok && x < w.nb; ++x) ok = load_block(x);
      }
      // Teardown: every copy issued must land before the CTA exits.
      if (n > 0) drain_wait(bar_afull, (n - 1) & 1, p.err);
      for (int x = (it > kS ? it - kS : 0); x < it; ++x) drain_wait(&bar_bfull[x % kS], (x / kS) & 1, p.err);
    }
  } else if (warp == kMmaWarp || warp == kAccWarp) {
    // ------------------------------------------------------------ MMA issuers
    constexpr uint32_t idesc_xy = make_idesc_f16(BF16, 128, kPN, false, false);
    constexpr uint32_t idesc_acc = make_idesc_f16(BF16, 128, D, false, true);
    const AccFlags accf = runtime_flags(S);
    bool ok = true;
    int i0 = 0;  // key blocks of the earlier items
    int n = 0;   // items
    if (warp == kMmaWarp) {
      const uint64_t a1_desc = make_sdesc(sA1, 16, 8 * GA::kRowBytes, GA::kSwz);
      const uint64_t a2_desc = make_sdesc(sA2, 16, 8 * GA::kRowBytes, GA::kSwz);
      for (int r = 0; ok; ++r) {
        const int k = item_at(r);
        if (k < 0) break;
        const Item w = decode(k);
        ok = warp_wait(bar_afull, n & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutMma);
        if (!ok) break;
        // Q and dO into TMEM (after the previous item's score products, which
        // read the columns they overwrite: the tensor core runs them in order).
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          tmem_cp_128x256b_warp(tmem + L::kColA1 + 8 * kk, desc_plus(a1_desc, kmajor_step_bytes<D, 128>(kk)));
          tmem_cp_128x256b_warp(tmem + L::kColA2 + 8 * kk, desc_plus(a2_desc, kmajor_step_bytes<D, 128>(kk)));
        }
        mma_commit_warp(bar_aempty);  // the shared-memory Q, dO are free once the copies land
        for (int x = 0; ok && x < w.nb; ++x) {
          const int i = i0 + x;
          const int st = i % kS;
          const int b = i % kB;
          ok = warp_wait<kSpinMma, kUnrollMma>(&bar_bfull[st], (i / kS) & 1, abort_flag, p.err, p.wait_ns,
                                               kErrTimeoutMma);
          if (ok && i >= kB)
            ok = warp_wait<kSpinMma, kUnrollMma>(&bar_accissued[b], ((i / kB) - 1) & 1, abort_flag, p.err,
                                                 p.wait_ns, kErrTimeoutMma);
          if (!ok) break;
          tc_fence_after();
          const uint32_t tb = tmem + 128u * b;
          const uint64_t b1 = make_sdesc(sB1 + st * GB::kTileBytes, 16, 8 * GB::kRowBytes, GB::kSwz);
          const uint64_t b2 = make_sdesc(sB2 + st * GB::kTileBytes, 16, 8 * GB::kRowBytes, GB::kSwz);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)  // X = S = Q K_j^T
            mma_ts_warp(tb, tmem + L::kColA1 + 8 * kk, desc_plus(b1, kmajor_step_bytes<D, kPN>(kk)), idesc_xy,
                        kk > 0 ? accf.on : accf.off);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)  // Y = dP = dO V_j^T
            mma_ts_warp(tb + 64, tmem + L::kColA2 + 8 * kk, desc_plus(b2, kmajor_step_bytes<D, kPN>(kk)), idesc_xy,
                        kk > 0 ? accf.on : accf.off);
          mma_commit_warp(&bar_xyfull[b]);
        }
        i0 += w.nb;
        ++n;
      }
      mma_commit_warp(&bar_drain[0]);
      drain_wait(&bar_drain[0], 0, p.err);
    } else {
      for (int r = 0; ok; ++r) {
        const int k = item_at(r);
        if (k < 0) break;
        const Item w = decode(k);
        for (int x = 0; ok && x < w.nb; ++x) {
          const int i = i0 + x;
          const int st = i % kS;
          const int b = i % kB;
          ok = warp_wait<kSpinMma, kUnrollMma>(&bar_pfull[i % kPFullBars], (i / kPFullBars) & 1, abort_flag, p.err,
                                               p.wait_ns, kErrTimeoutMma);
          // The item's first accumulation overwrites dQ: the previous item's
          // must have been read out.
          if (ok && x == 0 && n > 0)
            ok = warp_wait(bar_accfree, (n - 1) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutMma);
          if (!ok) break;
          tc_fence_after();
          const uint32_t tb = tmem + 128u * b;
          const uint64_t b1 = make_sdesc(sB1 + st * GB::kTileBytes, GB::kChunkBytes, 8 * GB::kRowBytes, GB::kSwz);
#pragma unroll
          for (int kk = 0; kk < kPN / 16; ++kk)  // dQ += dS K_j
            mma_ts_warp(tmem + L::kColAcc1, tb + 64 + packed_col(kk), desc_plus(b1, mnmajor_step_bytes<D>(kk)),
                        idesc_acc, (x > 0 || kk > 0) ? accf.on : accf.off);
          mma_commit_warp(&bar_empty[st]);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar_accissued[b]);
        }
        if (!ok) break;
        mma_commit_warp(bar_accfinal);  // the item's dQ is complete once this lands
        i0 += w.nb;
        ++n;
      }
      mma_commit_warp(&bar_drain[1]);
      drain_wait(&bar_drain[1], 0, p.err);
    }
  } else {
    // ------------------------------------------------------------ softmax-gradient warps 0-15
    const int g = warp >> 3;
    const int q4 = warp & 3;
    const int hf = (warp >> 2) & 1;
    const int col0 = 32 * hf;
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    const float sl2 = p.scale_log2;
    const float2 c2 = make_float2(sl2, sl2);
    constexpr int kParts = D >= 64 ? 4 : D / 16;
    constexpr int kEpiCols = D / kParts;
    const int col_part = warp >> 2;
    bool alive = true;
    int i0 = 0;
    int n = 0;
    for (int r = 0; alive; ++r) {
      const int k = item_at(r);
      if (k < 0) break;
      const Item w = decode(k);
      const int my = w.own0 + q4 * 32 + lane;  // this thread's query
      const int64_t rowbase = static_cast<int64_t>(w.bh) * S;
      // This row's L2 = L * log2 e (rows past S: L2 = +inf, so P = 0 exactly)
      // and its Delta, from the Delta warp.
      const float my_l2 = my < S ? p.lse[rowbase + my] * kLog2e : INFINITY;
      if (!warp_wait(&bar_deltafull[n & 1], (n >> 1) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutSoftmax)) {
        alive = false;
        break;
      }
      const float my_delta = delta_buf[(n & 1) * 128 + q4 * 32 + lane];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_deltafree[n & 1]);
      // This group's blocks of the item: global block indices i0 + x with (i0 + x) % 2 == g.
      for (int x = (g - i0) & 1; x < w.nb; x += kBwdGroups) {
        const int i = i0 + x;
        const int partner0 = x * kPN;
        if (!warp_wait(&bar_xyfull[i % kB], (i / kB) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutSoftmax)) {
          alive = false;
          break;
        }
        tc_fence_after();
        const uint32_t tX = tmem + lane_base + 128u * (i % kB) + col0;
        const uint32_t tY = tX + 64;
        const int lim = my - partner0 - col0;
        if (p.causal && partner0 + kPN - 1 > w.own0)  // the diagonal blocks: keys after the query masked
          grad_block<BF16, false, true>(tX, tY, nullptr, nullptr, c2, my_l2, my_delta, lim);
        else
          grad_block<BF16, false, false>(tX, tY, nullptr, nullptr, c2, my_l2, my_delta, lim);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_pfull[i % kPFullBars]);
      }
      if (!alive) break;
      // ---------------------------------------------------------- epilogue of the item
      if (!warp_wait(bar_accfinal, n & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutSoftmax)) {
        alive = false;
        break;
      }
      tc_fence_after();
      if (col_part < kParts) {
        const int c_begin = col_part * kEpiCols;
        const bool row_ok = my < S;
        const size_t off = static_cast<size_t>(rowbase + (row_ok ? my : 0)) * D;
        const uint32_t t_acc = tmem + lane_base;
        elem_t* dq_row = reinterpret_cast<elem_t*>(p.dq) + off;
#pragma unroll
        for (int cc = c_begin; cc < c_begin + kEpiCols; cc += 16) {
          uint32_t v16[16];
          tmem_ld16(t_acc + L::kColAcc1 + cc, v16);
          if (row_ok) store_row16<BF16>(dq_row + cc, v16, p.scale);
        }
      }
      // dQ is read: the next item's accumulation may overwrite it.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_accfree);
      i0 += w.nb;
      ++n;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

// Persistent version of the dK/dV pass for fixed-length calls at D <= 64 with
// at most 32 partner blocks per work item on average (launch_dkdv_t decides):
// a grid of at most one CTA per SM, each running the pipeline of
// fa_bwd_main_kernel over a sequence of the per-tile grid's key tiles (work
// items, in that grid's launch order, dealt in a snake as in the persistent
// dQ pass).  Between items: the producer loads the next item's first partner
// blocks, then its K and V tiles as soon as the current item's last score
// products have read them (a_empty); the accumulation warp starts the next
// item's dV, dK once all 16 softmax-gradient warps have read the current ones
// out of TMEM (acc_free).  The per-block steps run slower inside this
// kernel's item loops than in the per-tile kernel, so it pays only while the
// per-item overlap outweighs that: measured (whole backward, causal fp16 D64)
// B8 H16 S1024 111 -> 101 us, B4 H16 S2048 147 -> 139 us, B4 H16 S4096 417 ->
// 411 us, but B2 H16 S8192 703 -> 724 us and grouped K/V heads at S4096
// (hpc 2 or 4 query heads per item) 5-7 % slower.
template <int D, bool BF16>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_dkdvp_kernel(const __grid_constant__ CUtensorMap tm_a1, const __grid_constant__ CUtensorMap tm_a2,
                        const __grid_constant__ CUtensorMap tm_b1, const __grid_constant__ CUtensorMap tm_b2,
                        const BwdParams p, int gx, int n_items) {
  using L = BwdLayout<D>;
  static_assert(D <= 64, "persistent dK/dV pass: D <= 64");
  using GA = typename L::GA;
  using GB = typename L::GB;
  using elem_t = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  constexpr int kPN = kPartnerRows;
  constexpr int kS = L::kStages;
  constexpr int kB = L::kXYBufs;
  // Barrier tests before blocking as in fa_bwd_main_kernel's dK/dV pass, but
  // not unrolled: this kernel's longer code ran faster with the small loops
  // (c2 242 -> 234 us).
  constexpr int kSpinMma = 64;
  constexpr int kSpinOther = 64;
  constexpr int kUnrollMma = 1;
  constexpr int kUnrollOther = 1;
  constexpr int kPreBlocks = 4;  // partner blocks of the next item loaded before its resident tiles

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kOffBar);
  uint64_t* bar_afull = bars;
  uint64_t* bar_bfull = bars + 1;
  uint64_t* bar_empty = bar_bfull + kS;
  uint64_t* bar_xyfull = bar_empty + kS;         // [buffers]
  uint64_t* bar_accissued = bar_xyfull + kB;     // [buffers] accumulation reading it issued
  uint64_t* bar_pfull = bar_accissued + kB;      // [4] block i's P, dS stored: bar_pfull[i % 4]
  uint64_t* bar_accfinal = bar_pfull + kPFullBars;
  uint64_t* bar_drain = bar_accfinal + 1;        // [2] one per MMA warp
  uint64_t* bar_aempty = bar_drain + 2;          // the item's last score products (last reads of A1, A2) done
  uint64_t* bar_accfree = bar_aempty + 1;        // the item's accumulators read out by all 16 warps
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);
  float* vecs = reinterpret_cast<float*>(smem + L::kOffVec);

  const int warp = warp_index();
  const int lane = threadIdx.x & 31;
  const int S = p.S;
  const int nt = p.n_tiles;
  const int np = (S + kPN - 1) / kPN;
  const int hpc = p.group / p.kv_splits;  // query heads per CTA share of a K/V head
  const int gy = nt;
  const int P = static_cast<int>(gridDim.x);
  const int c = static_cast<int>(blockIdx.x);
  auto item_at = [&](int r) -> int {
    const int k = r * P + ((r & 1) ? (P - 1 - c) : c);
    return k < n_items ? k : -1;
  };
  // One work item: the tile the non-persistent grid's CTA number k took.
  struct Item {
    int bh, kv_part, pz0, own0, first, nper, niter;
  };
  auto decode = [&](int k) -> Item {
    int cx, cy;
    if (p.causal) {  // x fastest: every head's heaviest tile first
      cy = k / gx;
      cx = k - cy * gx;
    } else {         // y fastest: one head's tiles in a row
      cx = k / gy;
      cy = k - cx * gy;
    }
    Item it;
    it.bh = cx / p.kv_splits;  // K/V head
    it.kv_part = cx - it.bh * p.kv_splits;
    it.pz0 = it.bh * p.group + it.kv_part * hpc;  // first partner (query) head
    it.own0 = cy * 128;
    it.first = p.causal ? it.own0 / kPN : 0;
    it.nper = np - it.first;
    it.niter = hpc * it.nper;
    return it;
  };

  if (threadIdx.x == 0) {
    mbar_init(bar_afull, 1);
    for (int s = 0; s < kS; ++s) {
      mbar_init(&bar_bfull[s], 33);  // the TMA arrival + one cp.async arrival per producer lane
      mbar_init(&bar_empty[s], 1);
    }
    for (int b = 0; b < kB; ++b) {
      mbar_init(&bar_xyfull[b], 1);
      mbar_init(&bar_accissued[b], 1);
    }
    for (int b = 0; b < kPFullBars; ++b) mbar_init(&bar_pfull[b], 8);
    mbar_init(bar_accfinal, 1);
    mbar_init(&bar_drain[0], 1);
    mbar_init(&bar_drain[1], 1);
    mbar_init(bar_aempty, 1);
    mbar_init(bar_accfree, 16);  // one arrival per softmax-gradient warp
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
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

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_a1);
      prefetch_tmap(&tm_a2);
      prefetch_tmap(&tm_b1);
      prefetch_tmap(&tm_b2);
    }
    bool ok = true;
    int it = 0;  // partner blocks loaded so far
    int n = 0;   // items whose resident tiles were loaded
    for (int r = 0; ok; ++r) {
      const int k = item_at(r);
      if (k < 0) break;
      const Item w = decode(k);
      // Partner head and block of the next block to load, stepped without divisions.
      int pz = w.pz0, pblk = w.first;
      auto load_block = [&](int) -> bool {
        const int st = it % kS;
        const int use = it / kS;
        if (use > 0 && !warp_wait<kSpinOther, kUnrollOther>(&bar_empty[st], (use - 1) & 1, abort_flag, p.err,
                                                             p.wait_ns, kErrTimeoutLoad))
          return false;
        const int r0 = pblk * kPN;
        if (lane == 0) {
          mbar_arrive_expect_tx(&bar_bfull[st], 2 * GB::kTileBytes);
#pragma unroll
          for (int ch = 0; ch < GB::kChunks; ++ch) {
            tma_load_3d(smem + L::kOffB1 + st * GB::kTileBytes + ch * GB::kChunkBytes, &tm_b1, &bar_bfull[st],
                        ch * (GB::kRowBytes / 2), r0, pz);
            tma_load_3d(smem + L::kOffB2 + st * GB::kTileBytes + ch * GB::kChunkBytes, &tm_b2, &bar_bfull[st],
                        ch * (GB::kRowBytes / 2), r0, pz);
          }
        }
        // The block's L and Delta (partner queries past S read 0: their Q and
        // dO rows are zero-filled, so P dO and dS vanish there).  Delta may come
        // from the kernel just before this one (as in fa_bwd_main_kernel).
        if (it == 0) griddep_wait();
        float* v = vecs + st * 2 * kPN;
#pragma unroll
        for (int h = 0; h < kPN; h += 32) {
          const int q = r0 + h + lane;
          const int64_t src = static_cast<int64_t>(pz) * S + (q < S ? q : S - 1);
          cp_async_4(v + h + lane, p.lse + src, q < S);
          cp_async_4(v + kPN + h + lane, p.delta + src, q < S);
        }
        cp_async_mbar_arrive(&bar_bfull[st]);
        if (++pblk == w.first + w.nper) {
          pblk = w.first;
          ++pz;
        }
        ++it;
        return true;
      };
      const int pre = min(w.niter, kPreBlocks);
      for (int x = 0; ok && x < pre; ++x) ok = load_block(x);
      // The resident tiles, once the previous item's score products have read them.
      if (ok && n > 0)
        ok = warp_wait(bar_aempty, (n - 1) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutLoad);
      if (!ok) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar_afull, 2 * GA::kTileBytes);
#pragma unroll
        for (int ch = 0; ch < GA::kChunks; ++ch) {
          tma_load_3d(smem + L::kOffA1 + ch * GA::kChunkBytes, &tm_a1, bar_afull, ch * (GA::kRowBytes / 2), w.own0,
                      w.bh);
          tma_load_3d(smem + L::kOffA2 + ch * GA::kChunkBytes, &tm_a2, bar_afull, ch * (GA::kRowBytes / 2), w.own0,
                      w.bh);
        }
      }
      ++n;
      for (int x = pre; ok && x < w.niter; ++x) ok = load_block(x);
    }
    // Teardown: every copy issued must land before the CTA exits.
    if (lane == 0 && n > 0) drain_wait(bar_afull, (n - 1) & 1, p.err);
    for (int x = (it > kS ? it - kS : 0); x < it; ++x) drain_wait(&bar_bfull[x % kS], (x / kS) & 1, p.err);
  } else if (warp == kMmaWarp || warp == kAccWarp) {
    // ------------------------------------------------------------ MMA issuers
    constexpr uint32_t idesc_xy = make_idesc_f16(BF16, 128, kPN, false, false);
    constexpr uint32_t idesc_acc = make_idesc_f16(BF16, 128, D, false, true);
    const AccFlags accf = runtime_flags(S);
    bool ok = true;
    int i0 = 0;  // partner blocks of the earlier items
    int n = 0;   // items
    if (warp == kMmaWarp) {
      const uint64_t a1_desc = make_sdesc(sA1, 16, 8 * GA::kRowBytes, GA::kSwz);
      const uint64_t a2_desc = make_sdesc(sA2, 16, 8 * GA::kRowBytes, GA::kSwz);
      for (int r = 0; ok; ++r) {
        const int k = item_at(r);
        if (k < 0) break;
        const Item w = decode(k);
        ok = warp_wait(bar_afull, n & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutMma);
        if (!ok) break;
        for (int x = 0; ok && x < w.niter; ++x) {
          const int i = i0 + x;
          const int st = i % kS;
          const int b = i % kB;
          ok = warp_wait<kSpinMma, kUnrollMma>(&bar_bfull[st], (i / kS) & 1, abort_flag, p.err, p.wait_ns,
                                               kErrTimeoutMma);
          if (ok && i >= kB)
            ok = warp_wait<kSpinMma, kUnrollMma>(&bar_accissued[b], ((i / kB) - 1) & 1, abort_flag, p.err,
                                                 p.wait_ns, kErrTimeoutMma);
          if (!ok) break;
          tc_fence_after();
          const uint32_t tb = tmem + 128u * b;
          const uint64_t b1 = make_sdesc(sB1 + st * GB::kTileBytes, 16, 8 * GB::kRowBytes, GB::kSwz);
          const uint64_t b2 = make_sdesc(sB2 + st * GB::kTileBytes, 16, 8 * GB::kRowBytes, GB::kSwz);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)  // X = S^T = K Q_i^T
            mma_ss_warp(tb, desc_plus(a1_desc, kmajor_step_bytes<D, 128>(kk)),
                        desc_plus(b1, kmajor_step_bytes<D, kPN>(kk)), idesc_xy, kk > 0 ? accf.on : accf.off);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)  // Y = dP^T = V dO_i^T
            mma_ss_warp(tb + 64, desc_plus(a2_desc, kmajor_step_bytes<D, 128>(kk)),
                        desc_plus(b2, kmajor_step_bytes<D, kPN>(kk)), idesc_xy, kk > 0 ? accf.on : accf.off);
          mma_commit_warp(&bar_xyfull[b]);
        }
        if (!ok) break;
        mma_commit_warp(bar_aempty);  // the item's last reads of A1, A2 are issued
        i0 += w.niter;
        ++n;
      }
      mma_commit_warp(&bar_drain[0]);
      drain_wait(&bar_drain[0], 0, p.err);
    } else {
      for (int r = 0; ok; ++r) {
        const int k = item_at(r);
        if (k < 0) break;
        const Item w = decode(k);
        for (int x = 0; ok && x < w.niter; ++x) {
          const int i = i0 + x;
          const int st = i % kS;
          const int b = i % kB;
          ok = warp_wait<kSpinMma, kUnrollMma>(&bar_pfull[i % kPFullBars], (i / kPFullBars) & 1, abort_flag, p.err,
                                               p.wait_ns, kErrTimeoutMma);
          // The item's first accumulation overwrites the accumulators: the
          // previous item's must have been read out.
          if (ok && x == 0 && n > 0)
            ok = warp_wait(bar_accfree, (n - 1) & 1, abort_flag, p.err, p.wait_ns, kErrTimeoutMma);
          if (!ok) break;
          tc_fence_after();
          const uint32_t tb = tmem + 128u * b;
          const uint64_t b1 = make_sdesc(sB1 + st * GB::kTileBytes, GB::kChunkBytes, 8 * GB::kRowBytes, GB::kSwz);
          const uint64_t b2 = make_sdesc(sB2 + st * GB::kTileBytes, GB::kChunkBytes, 8 * GB::kRowBytes, GB::kSwz);
#pragma unroll
          for (int kk = 0; kk < kPN / 16; ++kk)  // dV += P^T dO_i
            mma_ts_warp(tmem + L::kColAcc1, tb + packed_col(kk), desc_plus(b2, mnmajor_step_bytes<D>(kk)), idesc_acc,
                        (x > 0 || kk > 0) ? accf.on : accf.off);
#pragma unroll
          for (int kk = 0; kk < kPN / 16; ++kk)  // dK += dS^T Q_i
            mma_ts_warp(tmem + L::kColAcc2, tb + 64 + packed_col(kk), desc_plus(b1, mnmajor_step_bytes<D>(kk)),
                        idesc_acc, (x > 0 || kk > 0) ? accf.on : accf.off);
          mma_commit_warp(&bar_empty[st]);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar_accissued[b]);
        }
        if (!ok) break;
        mma_commit_warp(bar_accfinal);  // the item's accumulators are complete once this lands
        i0 += w.niter;
        ++n;
      }
      mma_commit_warp(&bar_drain[1]);
      drain_wait(&bar_drain[1], 0, p.err);
    }
  } else {
    // ------------------------------------------------------------ softmax-gradient warps 0-15
    const int g = warp >> 3;
    const int q4 = warp & 3;
    const int hf = (warp >> 2) & 1;
    const int col0 = 32 * hf;
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    const float sl2 = p.scale_log2;
    const float2 c2 = make_float2(sl2, sl2);
    constexpr int kParts = D >= 64 ? 4 : D / 16;
    constexpr int kEpiCols = D / kParts;
    const int col_part = warp >> 2;
    bool alive = true;
    int i0 = 0;
    int n = 0;
    for (int r = 0; alive; ++r) {
      const int k = item_at(r);
      if (k < 0) break;
      const Item w = decode(k);
      const int my = w.own0 + q4 * 32 + lane;  // this thread's key
      const int64_t rowbase = static_cast<int64_t>(w.bh) * S;
      // This group's blocks of the item: global block indices i0 + x with (i0 + x) % 2 == g.
      const int x0 = (g - i0) & 1;
      int pi = x0;  // x modulo nper (the partner block within its head), stepped without divisions
      if (pi >= w.nper) pi -= w.nper;
      for (int x = x0; x < w.niter; x += kBwdGroups) {
        const int i = i0 + x;
        const int st = i % kS;
        const int partner0 = (w.first + pi) * kPN;
        pi += kBwdGroups;
        while (pi >= w.nper) pi -= w.nper;
        bool ok = warp_wait<kSpinOther, kUnrollOther>(&bar_bfull[st], (i / kS) & 1, abort_flag, p.err, p.wait_ns,
                                                      kErrTimeoutSoftmax);
        ok = ok && warp_wait<kSpinOther, kUnrollOther>(&bar_xyfull[i % kB], (i / kB) & 1, abort_flag, p.err,
                                                       p.wait_ns, kErrTimeoutSoftmax);
        if (!ok) {
          alive = false;
          break;
        }
        tc_fence_after();
        const uint32_t tX = tmem + lane_base + 128u * (i % kB) + col0;
        const uint32_t tY = tX + 64;
        const float* lv = vecs + st * 2 * kPN + col0;
        const float* dv = lv + kPN;
        // Diagonal blocks: partner queries before this key are masked.
        const int lim0 = w.own0 + q4 * 32 - partner0 - col0;
        if (p.causal && partner0 < w.own0 + 128)
          grad_block_kv<BF16, true>(tX, tY, lv, dv, c2, lim0);
        else
          grad_block_kv<BF16, false>(tX, tY, lv, dv, c2, lim0);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_pfull[i % kPFullBars]);
      }
      if (!alive) break;
      // ---------------------------------------------------------- epilogue of the item
      if (!warp_wait<kSpinOther, kUnrollOther>(bar_accfinal, n & 1, abort_flag, p.err, p.wait_ns,
                                               kErrTimeoutSoftmax)) {
        alive = false;
        break;
      }
      tc_fence_after();
      if (col_part < kParts) {
        const int c_begin = col_part * kEpiCols;
        const bool row_ok = my < S;
        const int64_t orow = rowbase + (row_ok ? my : 0);
        const size_t off = static_cast<size_t>(orow) * D;
        const uint32_t t_acc = tmem + lane_base;
        if (p.kv_splits == 1) {
          elem_t* dv_row = reinterpret_cast<elem_t*>(p.dv) + off;
          elem_t* dk_row = reinterpret_cast<elem_t*>(p.dk) + off;
#pragma unroll
          for (int cc = c_begin; cc < c_begin + kEpiCols; cc += 16) {
            uint32_t v16[16];
            tmem_ld16(t_acc + L::kColAcc1 + cc, v16);
            if (row_ok) store_row16<BF16>(dv_row + cc, v16, 1.f);
            tmem_ld16(t_acc + L::kColAcc2 + cc, v16);
            if (row_ok) store_row16<BF16>(dk_row + cc, v16, p.scale);
          }
        } else {
          // This CTA's share of the group: fp32 rows [dV | scale * dK] of partial kv_part.
          const int64_t n_rows = static_cast<int64_t>(p.BH / p.group) * S;
          float* prow = p.dkv_part + ((static_cast<int64_t>(w.kv_part) * n_rows + orow) * (2 * D));
#pragma unroll
          for (int cc = c_begin; cc < c_begin + kEpiCols; cc += 16) {
            uint32_t v16[16];
            tmem_ld16(t_acc + L::kColAcc1 + cc, v16);
            if (row_ok) store_row16_f32(prow + cc, v16, 1.f);
            tmem_ld16(t_acc + L::kColAcc2 + cc, v16);
            if (row_ok) store_row16_f32(prow + D + cc, v16, p.scale);
          }
        }
      }
      // The accumulators are read: the next item's accumulation may overwrite them.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_accfree);
      i0 += w.niter;
      ++n;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}


namespace {

template <int D, bool BF16>
cudaError_t launch_pre_t(const BwdParams& p, int64_t rows, cudaStream_t stream) {
  const int64_t threads = rows * (D / 8);
  const int64_t blocks = (threads + 255) / 256;
  const int grid = static_cast<int>(blocks < 152 * 16 ? blocks : 152 * 16);
  fa_bwd_preprocess_kernel<D, BF16><<<grid, 256, 0, stream>>>(p, rows);
  return cudaGetLastError();
}

// Launches `kern`; with `dependent`, as a programmatic dependent launch of the
// kernel before it on `stream`: its CTAs may start while that kernel's last
// CTAs still run, and it waits (griddep_wait) before reading that kernel's output.
template <typename... Params, typename... Args>
cudaError_t launch_kernel(void (*kern)(Params...), dim3 grid, int threads, int smem, cudaStream_t stream,
                          bool dependent, const Args&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = dependent ? attr : nullptr;
  cfg.numAttrs = dependent ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int D, bool BF16, bool KV_OUTER, bool GENERAL>
cudaError_t launch_main_t(const CUtensorMap& a1, const CUtensorMap& a2, const CUtensorMap& b1,
                          const CUtensorMap& b2, const BwdParams& p, cudaStream_t stream, bool dependent = false) {
  using L = BwdLayout<D>;
  auto kern = fa_bwd_main_kernel<D, BF16, KV_OUTER, GENERAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
  if (e != cudaSuccess) return e;
  // dK/dV pass: kv_splits CTAs per (K/V head, key tile); dQ pass: one per (query head, query tile).
  dim3 grid(KV_OUTER ? p.BH / p.group * p.kv_splits : p.BH, p.n_tiles);
  return launch_kernel(kern, grid, kBwdThreads, L::kSmemBytes, stream, dependent, a1, a2, b1, b2, p);
}

int bwd_sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      n = v;
    if (n <= 0) n = 1;
  }
  return n;
}

template <int D, bool BF16>
cudaError_t launch_dq_persistent_t(const CUtensorMap& a1, const CUtensorMap& a2, const CUtensorMap& b1,
                                   const CUtensorMap& b2, const BwdParams& p, cudaStream_t stream) {
  constexpr int kSmem = DqpLayout<D>::kSmemBytes;
  auto kern = fa_bwd_dqp_kernel<D, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  // Work items: the query tiles of the non-persistent grid (B*H x n_tiles).
  const int64_t n_items = static_cast<int64_t>(p.BH) * p.n_tiles;
  if (n_items <= 0) return cudaSuccess;
  if (n_items > (1LL << 30)) return cudaErrorInvalidValue;
  const int grid = static_cast<int>(n_items < bwd_sm_count() ? n_items : bwd_sm_count());
  kern<<<grid, kDqpThreads, kSmem, stream>>>(a1, a2, b1, b2, p, static_cast<int>(n_items));
  return cudaGetLastError();
}

// The dQ pass: the persistent kernel for fixed-length calls at D <= 64 (measured at causal
// B4 H16 S4096 D64 185 -> 165 us, B1 H16 S16384 D64 547 -> 538 us); at D = 128 the per-tile
// grid (the persistent kernel was as fast at B2 H32 S8192, 1.6 % slower at B1 H8 S32768).
template <int D, bool BF16>
cudaError_t launch_dq_t(bool general, const BwdMaps& m, const BwdParams& p, cudaStream_t stream, bool dependent) {
  if (general) return launch_main_t<D, BF16, false, true>(m.q128, m.do128, m.k64, m.v64, p, stream, dependent);
  if constexpr (D <= 64)  // the persistent kernel: bwd_dq_computes_delta(D, false)
    return launch_dq_persistent_t<D, BF16>(m.q128, m.do128, m.k64, m.v64, p, stream);
  else
    return launch_main_t<D, BF16, false, false>(m.q128, m.do128, m.k64, m.v64, p, stream, dependent);
}

template <int D, bool BF16>
cudaError_t launch_dkdv_persistent_t(const CUtensorMap& a1, const CUtensorMap& a2, const CUtensorMap& b1,
                                     const CUtensorMap& b2, const BwdParams& p, cudaStream_t stream,
                                     bool dependent) {
  using L = BwdLayout<D>;
  auto kern = fa_bwd_dkdvp_kernel<D, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
  if (e != cudaSuccess) return e;
  // Work items: the key tiles of the per-tile grid (K/V heads x kv_splits x n_tiles).
  const int gx = p.BH / p.group * p.kv_splits;
  const int64_t n_items = static_cast<int64_t>(gx) * p.n_tiles;
  if (n_items <= 0) return cudaSuccess;
  if (n_items > (1LL << 30)) return cudaErrorInvalidValue;
  const int grid = static_cast<int>(n_items < bwd_sm_count() ? n_items : bwd_sm_count());
  return launch_kernel(kern, dim3(grid), kBwdThreads, L::kSmemBytes, stream, dependent, a1, a2, b1, b2, p, gx,
                       static_cast<int>(n_items));
}

// The dK/dV pass: the persistent kernel for fixed-length calls at D <= 64 whose items average at
// most 32 partner blocks (query heads per item x 64-row query blocks, halved under the causal
// mask); the per-tile grid otherwise.
template <int D, bool BF16>
cudaError_t launch_dkdv_t(bool general, const BwdMaps& m, const BwdParams& p, cudaStream_t stream,
                          bool dependent) {
  if (general) return launch_main_t<D, BF16, true, true>(m.k128, m.v128, m.q64, m.do64, p, stream, dependent);
  if constexpr (D <= 64) {
    const int64_t blocks = static_cast<int64_t>(p.group / p.kv_splits) * ((p.S + kPartnerRows - 1) / kPartnerRows);
    if ((p.causal ? blocks / 2 : blocks) <= 32)
      return launch_dkdv_persistent_t<D, BF16>(m.k128, m.v128, m.q64, m.do64, p, stream, dependent);
  }
  return launch_main_t<D, BF16, true, false>(m.k128, m.v128, m.q64, m.do64, p, stream, dependent);
}

template <int D, bool BF16>
cudaError_t launch_reduce_t(const BwdParams& p, int64_t rows, cudaStream_t stream) {
  const int64_t threads = rows * (2 * D / 8);
  const int64_t blocks = (threads + 255) / 256;
  const int grid = static_cast<int>(blocks < 152 * 8 ? blocks : 152 * 8);
  fa_bwd_dkv_reduce_kernel<D, BF16><<<grid, 256, 0, stream>>>(p, rows);
  return cudaGetLastError();
}

}  // namespace

int bwd_kv_splits(int64_t BHkv, int64_t n_tiles, int group) {
  constexpr int64_t kWant = 2 * 152;
  if (group <= 1) return 1;
  for (int s = 1; s < group; ++s)
    if (group % s == 0 && BHkv * n_tiles * s >= kWant) return s;
  return group;
}

#define FA_BWD_DISPATCH(CALL)                                   \
  switch (D) {                                                  \
    case 16: return bf16 ? CALL(16, true) : CALL(16, false);    \
    case 32: return bf16 ? CALL(32, true) : CALL(32, false);    \
    case 64: return bf16 ? CALL(64, true) : CALL(64, false);    \
    case 128: return bf16 ? CALL(128, true) : CALL(128, false); \
    default: return cudaErrorInvalidValue;                      \
  }

cudaError_t launch_bwd_preprocess(int D, bool bf16, const BwdParams& p, int64_t rows, cudaStream_t stream) {
#define FA_PRE(DD, BB) launch_pre_t<DD, BB>(p, rows, stream)
  FA_BWD_DISPATCH(FA_PRE)
#undef FA_PRE
}

cudaError_t launch_bwd_dkdv(int D, bool bf16, bool general, const BwdMaps& m, const BwdParams& p,
                            cudaStream_t stream, bool dependent) {
#define FA_DKDV(DD, BB) launch_dkdv_t<DD, BB>(general, m, p, stream, dependent)
  FA_BWD_DISPATCH(FA_DKDV)
#undef FA_DKDV
}

cudaError_t launch_bwd_dkv_reduce(int D, bool bf16, const BwdParams& p, int64_t rows, cudaStream_t stream) {
#define FA_RED(DD, BB) launch_reduce_t<DD, BB>(p, rows, stream)
  FA_BWD_DISPATCH(FA_RED)
#undef FA_RED
}

cudaError_t launch_bwd_dq(int D, bool bf16, bool general, const BwdMaps& m, const BwdParams& p,
                          cudaStream_t stream, bool dependent) {
#define FA_DQ(DD, BB) launch_dq_t<DD, BB>(general, m, p, stream, dependent)
  FA_BWD_DISPATCH(FA_DQ)
#undef FA_DQ
}

#undef FA_BWD_DISPATCH

bool bwd_dq_computes_delta(int D, bool general) { return !general && D <= 64; }

}  // namespace fa
