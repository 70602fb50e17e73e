// C-ABI entry points: argument validation, tensor-map encoding and launches.
// Nothing here computes attention; every arithmetic step runs in the kernels.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <atomic>
#include <cstring>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.cuh"
#include "sm103_ptx.cuh"

namespace fa {

// One error word per device; kernels receive its address.
static __device__ int g_fa_device_error = 0;

int* device_error_word() {
  static int* addr[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_fa_device_error) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<int*>(a);
  }
  return addr[dev];
}

// Limit of each pipeline wait in the kernels launched from now on.
static std::atomic<unsigned long long> g_wait_limit_ns{ptx::kWaitLimitNs};

unsigned long long wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

}  // namespace fa

// ---------------------------------------------------------------------------
// Scratch for fa_bwd_noalloc.  Some callers cannot allocate device memory at
// the point where they need the backward pass (a custom allocator that must
// not be re-entered, a memory pool that is already fully carved up, code
// running under a framework that forbids cudaMalloc on its hot path).  For
// them the backward's one scratch buffer, the fp32 row vector D, lives in this
// fixed array instead of a caller workspace.  Every GPU that loads the library
// holds it (8 MiB) until the process exits.
namespace fa {
constexpr int64_t kNoAllocMaxRows = int64_t(1) << 21;  // B*H*S rows: 2 Mi floats = 8 MiB
static __device__ __align__(256) float g_noalloc_delta[kNoAllocMaxRows];

// Device address of g_noalloc_delta on the current device.  In host code the
// array's name only stands for the symbol, so the address is looked up once
// per device (with that device current) and cached.
float* noalloc_delta_address(cudaError_t* err) {
  static float* addr[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* a = nullptr;
    *err = cudaGetSymbolAddress(&a, g_noalloc_delta);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = static_cast<float*>(a);
  }
  return addr[dev];
}
}  // namespace fa

namespace {

thread_local char g_detail[256] = "";

fa_status fail(fa_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
fa_status fail(fa_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_detail, sizeof(g_detail), fmt, ap);
  va_end(ap);
  return s;
}

// cuTensorMapEncodeTiled, fetched from the driver through the runtime so the
// library does not link against libcuda directly.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// [BH, S, D] 16-bit tensor as a 3-D map {D, S, BH}; box {row_bytes/2, box_rows, 1}.
// Rows past S read as zero.
fa_status encode_qkv_map(CUtensorMap* map, const void* base, bool bf16, int64_t D, int64_t S, int64_t BH,
                         const char* name, unsigned box_rows = 128) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const int rb = fa::row_bytes_for(static_cast<int>(D));
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D * 2), static_cast<cuuint64_t>(S * D * 2)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(rb / 2), static_cast<cuuint32_t>(box_rows), 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUtensorMapSwizzle swz = rb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                     : (rb == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
  CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "tensor map for %s: cuTensorMapEncodeTiled error %d", name, (int)r);
  return FA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fa_status check_common(int64_t B, int64_t H, int64_t S, int64_t D, float scale, fa_dtype dtype) {
  if (B < 0 || H < 0 || S < 0) return fail(FA_ERR_INVALID_ARG, "negative size: B=%lld H=%lld S=%lld",
                                           (long long)B, (long long)H, (long long)S);
  if (dtype != FA_FP16 && dtype != FA_BF16) return fail(FA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
  if (!std::isfinite(scale)) return fail(FA_ERR_INVALID_ARG, "scale must be finite");
  if (D != 16 && D != 32 && D != 64 && D != 128)
    return fail(FA_ERR_UNSUPPORTED, "head dimension D=%lld is not one of 16, 32, 64, 128", (long long)D);
  if (B > 0 && H > (int64_t(1) << 31) / B) return fail(FA_ERR_UNSUPPORTED, "B*H must be below 2^31");
  if (S >= (int64_t(1) << 31)) return fail(FA_ERR_UNSUPPORTED, "S must be below 2^31");
  if ((S + 127) / 128 > 65535) return fail(FA_ERR_UNSUPPORTED, "S=%lld exceeds 65535 tiles of 128", (long long)S);
  // element count must fit comfortably in 64-bit byte offsets
  if (B * H > 0 && S * D > (int64_t(1) << 60) / (B * H)) return fail(FA_ERR_UNSUPPORTED, "tensor too large");
  return FA_OK;
}

fa_status check_ptr(const void* p, const char* name) {
  if (!p) return fail(FA_ERR_INVALID_ARG, "%s is NULL", name);
  if (!aligned16(p)) return fail(FA_ERR_ALIGNMENT, "%s is not 16-byte aligned", name);
  return FA_OK;
}

fa_status from_cuda(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return FA_OK;
  return fail(FA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr float kLog2e = 1.4426950408889634f;

// Grouped heads: H_kv K/V heads, each shared by H / H_kv consecutive query
// heads.  H_kv = H is ordinary multi-head attention.
fa_status check_heads(int64_t H, int64_t H_kv) {
  if (H_kv < 0 || H_kv > H) return fail(FA_ERR_INVALID_ARG, "H_kv=%lld must lie in [0, H=%lld]",
                                        (long long)H_kv, (long long)H);
  if (H > 0 && (H_kv == 0 || H % H_kv != 0))
    return fail(FA_ERR_INVALID_ARG, "H=%lld is not a multiple of H_kv=%lld", (long long)H, (long long)H_kv);
  if (H == 0 && H_kv != 0) return fail(FA_ERR_INVALID_ARG, "H_kv=%lld with H=0", (long long)H_kv);
  return FA_OK;
}

// One call's problem.  Fixed length: B entries of S rows, tensors [B, H(_kv), S, D].
// Packed batch (cu != nullptr): B samples over T = total tokens, tensors
// [T, H(_kv), D], S = the largest sample length; L is [H, T].
struct Shape {
  int64_t B, H, H_kv, S, D;
  const int32_t* cu;
  int64_t total;
  bool is_packed;
  int64_t win_left = -1, win_right = -1;  // window band; negative = unlimited
  bool packed() const { return is_packed; }
  // Kernel window sides (fa::kNoWindow = unlimited; causal fixes the right side at 0).
  int kernel_left() const { return win_left < 0 || win_left >= S ? fa::kNoWindow : static_cast<int>(win_left); }
  int kernel_right(bool causal) const {
    if (causal) return 0;
    return win_right < 0 || win_right >= S ? fa::kNoWindow : static_cast<int>(win_right);
  }
  // The general kernels serve packed batches and windows that cut the band;
  // fixed-length full/causal calls take the specialised ones.
  bool general(bool causal) const {
    return is_packed || kernel_left() != fa::kNoWindow || (!causal && kernel_right(false) != fa::kNoWindow);
  }
  int64_t q_rows() const { return packed() ? total * H : B * H * S; }      // rows of Q, O, dO, L, Delta
  int64_t kv_rows() const { return packed() ? total * H_kv : B * H_kv * S; }  // rows of K, V, dK, dV
  bool empty() const { return B * H == 0 || S == 0 || (packed() && total == 0); }
};

fa_status check_shape(const Shape& sh, float scale, fa_dtype dtype) {
  fa_status st = check_common(sh.B, sh.H, sh.S, sh.D, scale, dtype);
  if (st != FA_OK) return st;
  if ((st = check_heads(sh.H, sh.H_kv))) return st;
  if (sh.packed()) {
    if (sh.total < 0) return fail(FA_ERR_INVALID_ARG, "negative total tokens %lld", (long long)sh.total);
    if (sh.total >= (int64_t(1) << 31)) return fail(FA_ERR_UNSUPPORTED, "total tokens must be below 2^31");
    if (sh.H > 0 && sh.total * sh.H >= (int64_t(1) << 31))
      return fail(FA_ERR_UNSUPPORTED, "total tokens * H must be below 2^31");
    if (sh.cu && (reinterpret_cast<uintptr_t>(sh.cu) & 3u) != 0)
      return fail(FA_ERR_ALIGNMENT, "cu_seqlens is not 4-byte aligned");
  }
  return FA_OK;
}

// The tensor map of one input for the call's layout: {D, S, B*heads} (fixed
// length; rows past S read zero) or {D, heads, T} (packed; tokens past T read
// zero), box {row_bytes/2, box_rows, 1} or {row_bytes/2, 1, box_rows}.
fa_status encode_input(CUtensorMap* map, const void* base, bool bf16, const Shape& sh, int64_t heads,
                       const char* name, unsigned box_rows = 128) {
  if (!sh.packed()) return encode_qkv_map(map, base, bf16, sh.D, sh.S, sh.B * heads, name, box_rows);
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const int rb = fa::row_bytes_for(static_cast<int>(sh.D));
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(sh.D), static_cast<cuuint64_t>(heads),
                        static_cast<cuuint64_t>(sh.total)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(sh.D * 2), static_cast<cuuint64_t>(heads * sh.D * 2)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(rb / 2), 1u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUtensorMapSwizzle swz = rb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                     : (rb == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
  CUresult r = enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "tensor map for %s: cuTensorMapEncodeTiled error %d", name, (int)r);
  return FA_OK;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Split-KV: keys per shard (a multiple of 128) and shard count for a request of n splits.
void splitkv_layout(int64_t S, int64_t n, int* chunk, int* shards) {
  const int64_t per = (S + n - 1) / n;
  const int64_t c = ((per + 127) / 128) * 128;
  *chunk = static_cast<int>(c);
  *shards = static_cast<int>((S + c - 1) / c);
}

size_t splitkv_bytes(const Shape& sh, int shards) {
  return round256(static_cast<size_t>(shards) * static_cast<size_t>(sh.B * sh.H * sh.S) *
                  static_cast<size_t>(sh.D + 1) * sizeof(float));
}

// Forward; with split > 0 (general kernels, fixed layout) the keys are cut
// into shards whose fp32 partials go to `workspace`, then merged by L.
fa_status fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, const Shape& sh, int causal,
                   float scale, fa_dtype dtype, void* stream, int64_t split = 0, void* workspace = nullptr,
                   size_t workspace_bytes = 0) {
  g_detail[0] = 0;
  fa_status st = check_shape(sh, scale, dtype);
  if (st != FA_OK) return st;
  if (sh.empty()) return FA_OK;  // empty: nothing is read or written, pointers may be NULL
  if ((st = check_ptr(q, "q")) || (st = check_ptr(k, "k")) || (st = check_ptr(v, "v")) ||
      (st = check_ptr(o, "o")) || (st = check_ptr(lse, "lse")))
    return st;
  if (sh.packed() && !sh.cu) return fail(FA_ERR_INVALID_ARG, "cu_seqlens is NULL");
  int chunk = 0, shards = 1;
  if (split > 0) {
    splitkv_layout(sh.S, split, &chunk, &shards);
    const size_t need = splitkv_bytes(sh, shards);
    if (!workspace) return fail(FA_ERR_WORKSPACE, "workspace is NULL (%zu bytes needed)", need);
    if (workspace_bytes < need) return fail(FA_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", workspace_bytes, need);
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
      return fail(FA_ERR_ALIGNMENT, "workspace is not 256-byte aligned");
    if (static_cast<int64_t>(shards) * sh.B * sh.H > 65535 * 65535LL)
      return fail(FA_ERR_UNSUPPORTED, "too many shards");
    if (shards > 65535) return fail(FA_ERR_UNSUPPORTED, "at most 65535 shards");
  }
  const bool bf16 = dtype == FA_BF16;
  // Q in 128-row boxes (a CTA's own tiles); K and V in 64-row boxes.
  CUtensorMap tq, tk, tv;
  if ((st = encode_input(&tq, q, bf16, sh, sh.H, "q")) || (st = encode_input(&tk, k, bf16, sh, sh.H_kv, "k", 64)) ||
      (st = encode_input(&tv, v, bf16, sh, sh.H_kv, "v", 64)))
    return st;
  fa::FwdParams p;
  p.o = o;
  p.lse = lse;
  p.S = static_cast<int>(sh.S);
  p.cu_seqlens = sh.cu;
  p.heads = static_cast<int>(sh.H);
  p.total = static_cast<int>(sh.packed() ? sh.total : 0);
  const int rows_per_cta = fa::fwd_rows_per_cta(static_cast<int>(sh.D));
  p.n_m_tiles = static_cast<int>((sh.S + rows_per_cta - 1) / rows_per_cta);  // CTAs per (b, h)
  p.causal = causal ? 1 : 0;
  p.win_left = sh.kernel_left();
  p.win_right = sh.kernel_right(causal != 0);
  p.group = static_cast<int>(sh.H / sh.H_kv);
  p.kv_chunk = chunk;
  const int64_t rows = sh.B * sh.H * sh.S;
  p.o_part = split > 0 ? static_cast<float*>(workspace) : nullptr;
  p.lse_part = split > 0 ? static_cast<float*>(workspace) + static_cast<size_t>(shards) * rows * sh.D : nullptr;
  p.scale_log2 = scale * kLog2e;
  p.err = fa::device_error_word();
  if (!p.err) return fail(FA_ERR_CUDA, "cannot resolve the device error word on the current device");
  p.wait_ns = fa::wait_limit_ns();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = from_cuda(fa::launch_fwd(static_cast<int>(sh.D), bf16, split > 0 || sh.general(causal != 0), tq, tk, tv,
                                     p, static_cast<int>(sh.B * sh.H), s),
                      "forward launch")))
    return st;
  if (split > 0)
    return from_cuda(fa::launch_merge_lse(static_cast<int>(sh.D), bf16, p.o_part, p.lse_part, shards, rows, o, lse, s),
                     "split-KV merge launch");
  return FA_OK;
}

// Backward workspace: the fp32 row vector Delta of every query row, then, when
// the dK/dV pass splits a K/V head's query heads over several CTAs, their fp32
// partial [dV | dK] rows.  Heads must already be validated (H_kv divides H).
size_t bwd_workspace_layout(const Shape& sh, int* splits, size_t* delta_bytes) {
  *splits = 1;
  *delta_bytes = 0;
  if (sh.B <= 0 || sh.H <= 0 || sh.S <= 0 || sh.H_kv <= 0 || (sh.packed() && sh.total <= 0)) return 0;
  *delta_bytes = round256(static_cast<size_t>(sh.q_rows()) * sizeof(float));
  *splits = fa::bwd_kv_splits(sh.B * sh.H_kv, (sh.S + 127) / 128, static_cast<int>(sh.H / sh.H_kv));
  if (*splits == 1) return *delta_bytes;
  return *delta_bytes + round256(static_cast<size_t>(*splits) * static_cast<size_t>(sh.kv_rows()) *
                                 static_cast<size_t>(2 * sh.D) * sizeof(float));
}

fa_status bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                   void* dq, void* dk, void* dv, const Shape& sh, int causal, float scale, fa_dtype dtype,
                   void* workspace, size_t workspace_bytes, void* stream, void* const* marks) {
  g_detail[0] = 0;
  fa_status st = check_shape(sh, scale, dtype);
  if (st != FA_OK) return st;
  if (sh.empty()) return FA_OK;  // empty: nothing is read or written, pointers may be NULL
  if ((st = check_ptr(q, "q")) || (st = check_ptr(k, "k")) || (st = check_ptr(v, "v")) ||
      (st = check_ptr(o, "o")) || (st = check_ptr(dout, "dout")) || (st = check_ptr(lse, "lse")) ||
      (st = check_ptr(dq, "dq")) || (st = check_ptr(dk, "dk")) || (st = check_ptr(dv, "dv")))
    return st;
  if (sh.packed() && !sh.cu) return fail(FA_ERR_INVALID_ARG, "cu_seqlens is NULL");
  int splits = 1;
  size_t delta_bytes = 0;
  const size_t need = bwd_workspace_layout(sh, &splits, &delta_bytes);
  if (!workspace) return fail(FA_ERR_WORKSPACE, "workspace is NULL (%zu bytes needed)", need);
  if (workspace_bytes < need)
    return fail(FA_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", workspace_bytes, need);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(FA_ERR_ALIGNMENT, "workspace is not 256-byte aligned");
  const bool bf16 = dtype == FA_BF16;
  fa::BwdMaps maps;
  if ((st = encode_input(&maps.q128, q, bf16, sh, sh.H, "q")) ||
      (st = encode_input(&maps.k128, k, bf16, sh, sh.H_kv, "k")) ||
      (st = encode_input(&maps.v128, v, bf16, sh, sh.H_kv, "v")) ||
      (st = encode_input(&maps.do128, dout, bf16, sh, sh.H, "dout")) ||
      (st = encode_input(&maps.q64, q, bf16, sh, sh.H, "q", 64)) ||
      (st = encode_input(&maps.k64, k, bf16, sh, sh.H_kv, "k", 64)) ||
      (st = encode_input(&maps.v64, v, bf16, sh, sh.H_kv, "v", 64)) ||
      (st = encode_input(&maps.do64, dout, bf16, sh, sh.H, "dout", 64)))
    return st;
  fa::BwdParams p;
  p.o = o;
  p.dout = dout;
  p.lse = lse;
  p.delta = static_cast<float*>(workspace);
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.S = static_cast<int>(sh.S);
  p.cu_seqlens = sh.cu;
  p.heads = static_cast<int>(sh.H);
  p.total = static_cast<int>(sh.packed() ? sh.total : 0);
  p.BH = static_cast<int>(sh.B * sh.H);
  p.group = static_cast<int>(sh.H / sh.H_kv);
  p.kv_splits = splits;
  p.dkv_part = splits > 1 ? reinterpret_cast<float*>(static_cast<char*>(workspace) + delta_bytes) : nullptr;
  p.n_tiles = static_cast<int>((sh.S + 127) / 128);
  p.causal = causal ? 1 : 0;
  p.win_left = sh.kernel_left();
  p.win_right = sh.kernel_right(causal != 0);
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  p.err = fa::device_error_word();
  if (!p.err) return fail(FA_ERR_CUDA, "cannot resolve the device error word on the current device");
  p.wait_ns = fa::wait_limit_ns();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int Di = static_cast<int>(sh.D);
  const int64_t q_rows = sh.q_rows(), kv_rows = sh.kv_rows();
  auto mark = [&](int i) -> fa_status {
    if (!marks || !marks[i]) return FA_OK;
    return from_cuda(cudaEventRecord(static_cast<cudaEvent_t>(marks[i]), s), "event record");
  };
  const bool general = sh.general(causal != 0);
  const bool fused_delta = fa::bwd_dq_computes_delta(Di, general);
  // Delta then dK/dV then dQ; or, when the dQ kernel computes Delta, dQ then dK/dV.
  if ((st = mark(0))) return st;
  if (fused_delta) {
    if ((st = from_cuda(fa::launch_bwd_dq(Di, bf16, general, maps, p, s, false), "backward dQ launch"))) return st;
  } else if ((st = from_cuda(fa::launch_bwd_preprocess(Di, bf16, p, q_rows, s), "backward preprocess launch"))) {
    return st;
  }
  if ((st = mark(1))) return st;
  // The second and third kernels are programmatic dependent launches: their
  // first CTAs start as the previous kernel's last ones finish.
  if ((st = from_cuda(fa::launch_bwd_dkdv(Di, bf16, general, maps, p, s, true), "backward dK/dV launch")))
    return st;
  if (splits > 1 &&
      (st = from_cuda(fa::launch_bwd_dkv_reduce(Di, bf16, p, kv_rows, s), "backward dK/dV reduce launch")))
    return st;
  if ((st = mark(2))) return st;
  if (!fused_delta &&
      (st = from_cuda(fa::launch_bwd_dq(Di, bf16, general, maps, p, s, true), "backward dQ launch")))
    return st;
  return mark(3);
}

Shape fixed(int64_t B, int64_t H, int64_t H_kv, int64_t S, int64_t D) {
  return Shape{B, H, H_kv, S, D, nullptr, 0, false};
}

Shape windowed(int64_t B, int64_t H, int64_t H_kv, int64_t S, int64_t D, int64_t left, int64_t right) {
  Shape sh{B, H, H_kv, S, D, nullptr, 0, false};
  sh.win_left = left;
  sh.win_right = right;
  return sh;
}

Shape packed(const int32_t* cu, int64_t batch, int64_t max_seqlen, int64_t total, int64_t H, int64_t H_kv,
             int64_t D) {
  return Shape{batch, H, H_kv, max_seqlen, D, cu, total, true};
}

}  // namespace

extern "C" {

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H, int64_t S,
                 int64_t D, int causal, float scale, fa_dtype dtype, void* stream) {
  return fwd_impl(q, k, v, o, lse, fixed(B, H, H, S, D), causal, scale, dtype, stream);
}

fa_status fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
                     int64_t H_kv, int64_t S, int64_t D, int causal, float scale, fa_dtype dtype, void* stream) {
  return fwd_impl(q, k, v, o, lse, fixed(B, H, H_kv, S, D), causal, scale, dtype, stream);
}

fa_status fa_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
                        int64_t H_kv, int64_t S, int64_t D, int causal, int64_t window_left, int64_t window_right,
                        float scale, fa_dtype dtype, void* stream) {
  return fwd_impl(q, k, v, o, lse, windowed(B, H, H_kv, S, D, window_left, window_right), causal, scale, dtype,
                  stream);
}

fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
                         int64_t H_kv, int64_t S, int64_t D, int causal, int64_t num_splits, float scale,
                         fa_dtype dtype, void* workspace, size_t workspace_bytes, void* stream) {
  if (num_splits < 1) {
    g_detail[0] = 0;
    return fail(FA_ERR_INVALID_ARG, "num_splits=%lld must be at least 1", (long long)num_splits);
  }
  return fwd_impl(q, k, v, o, lse, fixed(B, H, H_kv, S, D), causal, scale, dtype, stream, num_splits, workspace,
                  workspace_bytes);
}

size_t fa_fwd_splitkv_workspace_size(int64_t B, int64_t H, int64_t S, int64_t D, int64_t num_splits) {
  if (B <= 0 || H <= 0 || S <= 0 || num_splits < 1) return 0;
  int chunk = 0, shards = 1;
  splitkv_layout(S, num_splits, &chunk, &shards);
  return splitkv_bytes(fixed(B, H, H, S, D), shards);
}

int64_t fa_splitkv_num_splits(int64_t B, int64_t H, int64_t S, int64_t D) {
  // Enough shards to give every SM of a 152-SM GPU two CTAs, no more than one
  // shard per 128 keys.
  if (B <= 0 || H <= 0 || S <= 0 || (D != 16 && D != 32 && D != 64 && D != 128)) return 1;
  const int64_t rows_per_cta = fa::fwd_rows_per_cta(static_cast<int>(D));
  const int64_t ctas = B * H * ((S + rows_per_cta - 1) / rows_per_cta);
  const int64_t want = (2 * 152 + ctas - 1) / ctas;
  const int64_t cap = (S + 127) / 128;
  return want < 1 ? 1 : (want > cap ? cap : want);
}

fa_status fa_merge_lse(const float* o_part, const float* lse_part, void* o, float* lse, int64_t shards,
                       int64_t rows, int64_t D, fa_dtype dtype, void* stream) {
  g_detail[0] = 0;
  if (shards < 1 || rows < 0) return fail(FA_ERR_INVALID_ARG, "shards must be >= 1 and rows >= 0");
  if (dtype != FA_FP16 && dtype != FA_BF16) return fail(FA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
  if (D != 16 && D != 32 && D != 64 && D != 128)
    return fail(FA_ERR_UNSUPPORTED, "head dimension D=%lld is not one of 16, 32, 64, 128", (long long)D);
  if (shards > (int64_t(1) << 31) || (rows > 0 && shards > (int64_t(1) << 60) / (rows * (D + 1))))
    return fail(FA_ERR_UNSUPPORTED, "partials too large");
  if (rows == 0) return FA_OK;
  fa_status st;
  if ((st = check_ptr(o_part, "o_part")) || (st = check_ptr(lse_part, "lse_part")) || (st = check_ptr(o, "o")) ||
      (st = check_ptr(lse, "lse")))
    return st;
  return from_cuda(fa::launch_merge_lse(static_cast<int>(D), dtype == FA_BF16, o_part, lse_part,
                                        static_cast<int>(shards), rows, o, lse, static_cast<cudaStream_t>(stream)),
                   "merge launch");
}

fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                        const int32_t* cu_seqlens, int64_t batch, int64_t max_seqlen, int64_t total, int64_t H,
                        int64_t H_kv, int64_t D, int causal, float scale, fa_dtype dtype, void* stream) {
  return fwd_impl(q, k, v, o, lse, packed(cu_seqlens, batch, max_seqlen, total, H, H_kv, D), causal, scale, dtype,
                  stream);
}

size_t fa_bwd_workspace_size(int64_t B, int64_t H, int64_t S, int64_t D) {
  int splits = 1;
  size_t delta_bytes = 0;
  if (B < 0 || H < 0 || S < 0) return 0;
  return bwd_workspace_layout(fixed(B, H, H, S, D), &splits, &delta_bytes);
}

size_t fa_bwd_gqa_workspace_size(int64_t B, int64_t H, int64_t H_kv, int64_t S, int64_t D) {
  if (B < 0 || S < 0 || H_kv <= 0 || H <= 0 || H % H_kv != 0) return 0;
  int splits = 1;
  size_t delta_bytes = 0;
  return bwd_workspace_layout(fixed(B, H, H_kv, S, D), &splits, &delta_bytes);
}

size_t fa_bwd_varlen_workspace_size(int64_t batch, int64_t max_seqlen, int64_t total, int64_t H, int64_t H_kv,
                                    int64_t D) {
  if (batch < 0 || max_seqlen < 0 || total < 0 || H_kv <= 0 || H <= 0 || H % H_kv != 0) return 0;
  int splits = 1;
  size_t delta_bytes = 0;
  return bwd_workspace_layout(packed(nullptr, batch, max_seqlen, total, H, H_kv, D), &splits, &delta_bytes);
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                 void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t S, int64_t D, int causal, float scale,
                 fa_dtype dtype, void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, fixed(B, H, H, S, D), causal, scale, dtype, workspace,
                  workspace_bytes, stream, nullptr);
}

fa_status fa_bwd_marked(const void* q, const void* k, const void* v, const void* o, const void* dout,
                        const float* lse, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t S, int64_t D,
                        int causal, float scale, fa_dtype dtype, void* workspace, size_t workspace_bytes,
                        void* stream, void* const* marks) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, fixed(B, H, H, S, D), causal, scale, dtype, workspace,
                  workspace_bytes, stream, marks);
}

fa_status fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                     void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t H_kv, int64_t S, int64_t D,
                     int causal, float scale, fa_dtype dtype, void* workspace, size_t workspace_bytes,
                     void* stream) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, fixed(B, H, H_kv, S, D), causal, scale, dtype, workspace,
                  workspace_bytes, stream, nullptr);
}

fa_status fa_bwd_gqa_marked(const void* q, const void* k, const void* v, const void* o, const void* dout,
                            const float* lse, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t H_kv,
                            int64_t S, int64_t D, int causal, float scale, fa_dtype dtype, void* workspace,
                            size_t workspace_bytes, void* stream, void* const* marks) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, fixed(B, H, H_kv, S, D), causal, scale, dtype, workspace,
                  workspace_bytes, stream, marks);
}

fa_status fa_bwd_window_marked(const void* q, const void* k, const void* v, const void* o, const void* dout,
                               const float* lse, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t H_kv,
                               int64_t S, int64_t D, int causal, int64_t window_left, int64_t window_right,
                               float scale, fa_dtype dtype, void* workspace, size_t workspace_bytes, void* stream,
                               void* const* marks) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, windowed(B, H, H_kv, S, D, window_left, window_right), causal,
                  scale, dtype, workspace, workspace_bytes, stream, marks);
}

fa_status fa_bwd_window(const void* q, const void* k, const void* v, const void* o, const void* dout,
                        const float* lse, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t H_kv,
                        int64_t S, int64_t D, int causal, int64_t window_left, int64_t window_right, float scale,
                        fa_dtype dtype, void* workspace, size_t workspace_bytes, void* stream) {
  return fa_bwd_window_marked(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, S, D, causal, window_left,
                              window_right, scale, dtype, workspace, workspace_bytes, stream, nullptr);
}

fa_status fa_bwd_varlen_marked(const void* q, const void* k, const void* v, const void* o, const void* dout,
                               const float* lse, void* dq, void* dk, void* dv, const int32_t* cu_seqlens,
                               int64_t batch, int64_t max_seqlen, int64_t total, int64_t H, int64_t H_kv, int64_t D,
                               int causal, float scale, fa_dtype dtype, void* workspace, size_t workspace_bytes,
                               void* stream, void* const* marks) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, packed(cu_seqlens, batch, max_seqlen, total, H, H_kv, D),
                  causal, scale, dtype, workspace, workspace_bytes, stream, marks);
}

fa_status fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dout,
                        const float* lse, void* dq, void* dk, void* dv, const int32_t* cu_seqlens, int64_t batch,
                        int64_t max_seqlen, int64_t total, int64_t H, int64_t H_kv, int64_t D, int causal,
                        float scale, fa_dtype dtype, void* workspace, size_t workspace_bytes, void* stream) {
  return fa_bwd_varlen_marked(q, k, v, o, dout, lse, dq, dk, dv, cu_seqlens, batch, max_seqlen, total, H, H_kv, D,
                              causal, scale, dtype, workspace, workspace_bytes, stream, nullptr);
}

fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                         const float* lse, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t S,
                         int64_t D, int causal, float scale, fa_dtype dtype, void* stream) {
  g_detail[0] = 0;
  fa_status st = check_common(B, H, S, D, scale, dtype);
  if (st != FA_OK) return st;
  const int64_t BH = B * H;
  if (BH == 0 || S == 0) return FA_OK;
  if (BH > fa::kNoAllocMaxRows / S)
    return fail(FA_ERR_UNSUPPORTED, "fa_bwd_noalloc: B*H*S = %lld rows exceeds its fixed scratch of %lld rows",
                (long long)(BH * S), (long long)fa::kNoAllocMaxRows);
  cudaError_t e = cudaSuccess;
  float* delta = fa::noalloc_delta_address(&e);
  if (!delta) return from_cuda(e, "fa_bwd_noalloc: address of the scratch array");
  // The same kernels as fa_bwd, with the scratch array as the workspace.
  // Every row's Delta is written (by the Delta kernel or the dQ pass) before it
  // is read, so nothing needs clearing.
  return fa_bwd_marked(q, k, v, o, dout, lse, dq, dk, dv, B, H, S, D, causal, scale, dtype, delta,
                       static_cast<size_t>(fa::kNoAllocMaxRows) * sizeof(float), stream, nullptr);
}

const char* fa_status_string(fa_status status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_ALIGNMENT: return "FA_ERR_ALIGNMENT";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
  }
  return "FA_ERR_UNKNOWN";
}

const char* fa_last_error_detail(void) { return g_detail; }

uint64_t fa_set_wait_limit_ns(uint64_t ns) {
  const unsigned long long v = ns == 0 ? fa::ptx::kWaitLimitNs : static_cast<unsigned long long>(ns);
  return static_cast<uint64_t>(fa::g_wait_limit_ns.exchange(v));
}

fa_status fa_check_device_errors(void* stream) {
  g_detail[0] = 0;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return from_cuda(e, "stream synchronize");
  int code = 0;
  e = cudaMemcpyFromSymbol(&code, fa::g_fa_device_error, sizeof(int));
  if (e != cudaSuccess) return from_cuda(e, "read device error word");
  if (code != 0) {
    const int zero = 0;
    cudaMemcpyToSymbol(fa::g_fa_device_error, &zero, sizeof(int));
    if (code == fa::kErrBadSeqlens)
      return fail(FA_ERR_INVALID_ARG, "cu_seqlens contradicts max_seqlen or the token count (checked on the device)");
    return fail(FA_ERR_TIMEOUT, "device pipeline wait timed out (code %d)", code);
  }
  return FA_OK;
}

}  // extern "C"
