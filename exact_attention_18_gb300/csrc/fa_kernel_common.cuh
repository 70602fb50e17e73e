// Helpers shared by the forward and backward kernels: shared-memory tile
// geometry, MMA operand descriptors for TMA-swizzled tiles, bounded waits
// that stay warp-uniform, and 16-bit packing.
#pragma once

#include <type_traits>

#include "fa_internal.cuh"
#include "sm103_ptx.cuh"

namespace fa {

// A [ROWS, D] tile of 16-bit elements as TMA writes it: `kChunks` column
// chunks of ROWS rows x kRowBytes, each swizzled at kRowBytes granularity.
template <int D, int ROWS = 128>
struct TileGeom {
  static constexpr int kRowBytes = D * 2 < 128 ? D * 2 : 128;
  static constexpr int kChunks = D * 2 / kRowBytes;
  static constexpr int kChunkBytes = ROWS * kRowBytes;
  static constexpr int kTileBytes = ROWS * D * 2;
  static constexpr uint32_t kSwz = ptx::swizzle_code_for(kRowBytes);
};

// Operand descriptor for K-step kk (16 elements along D) of a tile read
// K-major (rows = M or N, D contiguous).
template <int D, int ROWS = 128>
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile_addr, int kk) {
  using G = TileGeom<D, ROWS>;
  const int off = kk * 32;
  return ptx::make_sdesc(tile_addr + (off / G::kRowBytes) * G::kChunkBytes + (off % G::kRowBytes), 16,
                         8 * G::kRowBytes, G::kSwz);
}

// Operand descriptor for K-step kk (tile rows 16kk..16kk+15) of a tile read
// MN-major (the tile's D columns are the N dimension, its rows the K dimension).
template <int D, int ROWS = 128>
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t tile_addr, int kk) {
  using G = TileGeom<D, ROWS>;
  return ptx::make_sdesc(tile_addr + kk * 16 * G::kRowBytes, G::kChunkBytes, 8 * G::kRowBytes, G::kSwz);
}

// Byte offset of K-step kk inside a K-major tile (added to a base descriptor's
// start-address field as offset >> 4).
template <int D, int ROWS = 128>
__host__ __device__ constexpr uint32_t kmajor_step_bytes(int kk) {
  using G = TileGeom<D, ROWS>;
  return static_cast<uint32_t>(((kk * 32) / G::kRowBytes) * G::kChunkBytes + (kk * 32) % G::kRowBytes);
}
// Byte offset of K-step kk (16 tile rows) inside an MN-major tile.
template <int D>
__host__ __device__ constexpr uint32_t mnmajor_step_bytes(int kk) {
  return static_cast<uint32_t>(kk * 16 * TileGeom<D>::kRowBytes);
}
// A descriptor advanced by `bytes` (start address is in 16-byte units in the low bits).
__device__ __forceinline__ uint64_t desc_plus(uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); }

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// The warp's index within the CTA, read through a shuffle from lane 0 so the
// compiler knows it is the same in every lane.  Everything derived from it
// (tile index, TMEM addresses, shared-memory descriptors) then lives in
// uniform registers, which tcgen05 instructions take as operands directly;
// derived from threadIdx.x alone it is a per-lane value, and every MMA, TMEM
// load and store first copies its operands into uniform registers.  Measured:
// the D = 64 forward at causal B4 H16 S4096 took 152 us with threadIdx.x / 32,
// 133 us with this; the backward passes 277 / 214 us against 258 / 192 us.
__device__ __forceinline__ int warp_index() {
  return __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
}

// All 32 lanes wait; the outcome is made warp-uniform (any failure = failure),
// so the warp-collective tcgen05 loads and stores that follow never diverge.
template <int kSpin = 0, int kUnroll = 1>
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int* err,
                                          unsigned long long limit_ns, int code) {
  const bool ok = ptx::mbar_wait<kSpin, kUnroll>(bar, parity, abort, err, limit_ns, code);
  return __all_sync(0xffffffffu, ok);
}

// Bounded wait that ignores the abort flag: used at teardown for the CTA's
// own copies and MMAs, which complete without help from other warps.  Its
// limit is always kWaitLimitNs, whatever limit the pipeline waits have: the
// CTA must not exit while a copy into its shared memory is still in flight.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, int* err) {
  if (ptx::mbar_try_wait(bar, parity)) return;
  const unsigned long long t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer() - t0 > ptx::kWaitLimitNs) {
      ptx::record_error(err, kErrTimeoutDrain);
      return;
    }
  }
}

// Coordinates (x = head, y = tile) of this CTA in a (gridDim.x, gridDim.y)
// grid.  Without a causal mask every tile of a head costs the same, so the
// launch order is taken y-fastest: one head's tiles run as consecutive CTAs
// and the CTAs resident at one time stream the keys and values (or queries
// and output gradients) of a few heads, which stay in L2.  Under the causal
// mask the order stays x-fastest so that every head's heaviest tile comes
// before any lighter one.
__device__ __forceinline__ void cta_coords(bool y_fastest, int* x, int* y) {
  int cx = static_cast<int>(blockIdx.x), cy = static_cast<int>(blockIdx.y);
  if (y_fastest) {
    const int lin = cx + cy * static_cast<int>(gridDim.x);
    cx = lin / static_cast<int>(gridDim.y);
    cy = lin - cx * static_cast<int>(gridDim.y);
  }
  *x = cx;
  *y = cy;
}

// Packed batch: first token and length of sample b from cu_seqlens (read by
// every thread).  Returns false, and records kErrBadSeqlens, when the entries
// contradict the call (negative start, decreasing offsets, a sample longer
// than max_len, or one ending past `total` tokens); the caller then exits
// before touching any tensor.
__device__ __forceinline__ bool packed_sample(const int* cu, int b, int max_len, int total, int* err, int* tok0,
                                              int* len) {
  const int a = __ldg(cu + b);
  const int e = __ldg(cu + b + 1);
  *tok0 = a;
  *len = e - a;
  if (a < 0 || e < a || e - a > max_len || e > total) {
    if (threadIdx.x == 0) ptx::record_error(err, kErrBadSeqlens);
    return false;
  }
  return true;
}

// Named barrier among the `nthreads` threads (a multiple of 32) that use `id`.
__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Arrive at named barrier `id` (counted among `nthreads`) without waiting.
__device__ __forceinline__ void named_arrive(int id, int nthreads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Barrier over `nthreads` threads with id `id` that also returns the AND of
// every participant's `v`.
__device__ __forceinline__ bool named_sync_and(int id, int nthreads, bool v) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, %2, %3, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(out)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(nthreads)
      : "memory");
  return out != 0;
}

// Store 16 fp32 values (times `mul`) as 16 16-bit elements at dst (32 bytes).
template <bool BF16>
__device__ __forceinline__ void store_row16(void* dst, const uint32_t* v, float mul) {
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = pack2<BF16>(__uint_as_float(v[2 * i]) * mul, __uint_as_float(v[2 * i + 1]) * mul);
  uint4* d = reinterpret_cast<uint4*>(dst);
  d[0] = make_uint4(w[0], w[1], w[2], w[3]);
  d[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

// 16 fp32 values (TMEM words) times `mul` to 16 consecutive floats (64 bytes, 16-byte aligned).
__device__ __forceinline__ void store_row16_f32(float* dst, const uint32_t* v, float mul) {
  float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    d[i] = make_float4(__uint_as_float(v[4 * i]) * mul, __uint_as_float(v[4 * i + 1]) * mul,
                       __uint_as_float(v[4 * i + 2]) * mul, __uint_as_float(v[4 * i + 3]) * mul);
}

}  // namespace fa
