// C-ABI entry points: argument validation, tensor-map encoding and launches.
// Nothing here computes attention; every arithmetic step runs in the kernels.
#include <cmath>
#include <cstdarg>
#include <cstdio>
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

fa_status fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
                   int64_t H_kv, int64_t S, int64_t D, int causal, float scale, fa_dtype dtype, void* stream) {
  g_detail[0] = 0;
  fa_status st = check_common(B, H, S, D, scale, dtype);
  if (st != FA_OK) return st;
  if ((st = check_heads(H, H_kv))) return st;
  const int64_t BH = B * H;
  if (BH == 0 || S == 0) return FA_OK;  // empty: nothing is read or written, pointers may be NULL
  if ((st = check_ptr(q, "q")) || (st = check_ptr(k, "k")) || (st = check_ptr(v, "v")) ||
      (st = check_ptr(o, "o")) || (st = check_ptr(lse, "lse")))
    return st;
  const bool bf16 = dtype == FA_BF16;
  // Q in 128-row boxes (a CTA's own tiles); K and V in 64-row boxes.
  CUtensorMap tq, tk, tv;
  const int64_t BHkv = B * H_kv;
  if ((st = encode_qkv_map(&tq, q, bf16, D, S, BH, "q")) ||
      (st = encode_qkv_map(&tk, k, bf16, D, S, BHkv, "k", 64)) ||
      (st = encode_qkv_map(&tv, v, bf16, D, S, BHkv, "v", 64)))
    return st;
  fa::FwdParams p;
  p.o = o;
  p.lse = lse;
  p.S = static_cast<int>(S);
  const int rows_per_cta = fa::fwd_rows_per_cta(static_cast<int>(D));
  p.n_m_tiles = static_cast<int>((S + rows_per_cta - 1) / rows_per_cta);  // CTAs per (b, h)
  p.causal = causal ? 1 : 0;
  p.group = static_cast<int>(H / H_kv);
  p.scale_log2 = scale * kLog2e;
  p.err = fa::device_error_word();
  if (!p.err) return fail(FA_ERR_CUDA, "cannot resolve the device error word on the current device");
  return from_cuda(fa::launch_fwd(static_cast<int>(D), bf16, tq, tk, tv, p, static_cast<int>(BH),
                                  static_cast<cudaStream_t>(stream)),
                   "forward launch");
}

fa_status bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                   void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t H_kv, int64_t S, int64_t D,
                   int causal, float scale, fa_dtype dtype, void* workspace, size_t workspace_bytes,
                   void* stream, void* const* marks);

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Backward workspace: the fp32 row vector Delta of every query row, then, when
// the dK/dV pass splits a K/V head's query heads over several CTAs, their fp32
// partial [dV | dK] rows.  Sizes must already be validated (H_kv divides H).
size_t bwd_workspace_layout(int64_t B, int64_t H, int64_t H_kv, int64_t S, int64_t D, int* splits,
                            size_t* delta_bytes) {
  *splits = 1;
  *delta_bytes = 0;
  if (B <= 0 || H <= 0 || S <= 0 || H_kv <= 0) return 0;
  *delta_bytes = round256(static_cast<size_t>(B) * static_cast<size_t>(H) * static_cast<size_t>(S) * sizeof(float));
  *splits = fa::bwd_kv_splits(B * H_kv, (S + 127) / 128, static_cast<int>(H / H_kv));
  if (*splits == 1) return *delta_bytes;
  return *delta_bytes + round256(static_cast<size_t>(*splits) * static_cast<size_t>(B * H_kv) *
                                 static_cast<size_t>(S) * static_cast<size_t>(2 * D) * sizeof(float));
}

}  // namespace

extern "C" {

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H, int64_t S,
                 int64_t D, int causal, float scale, fa_dtype dtype, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, H, S, D, causal, scale, dtype, stream);
}

fa_status fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
                     int64_t H_kv, int64_t S, int64_t D, int causal, float scale, fa_dtype dtype, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, H, H_kv, S, D, causal, scale, dtype, stream);
}

size_t fa_bwd_workspace_size(int64_t B, int64_t H, int64_t S, int64_t D) {
  int splits = 1;
  size_t delta_bytes = 0;
  return bwd_workspace_layout(B, H, H, S, D, &splits, &delta_bytes);
}

size_t fa_bwd_gqa_workspace_size(int64_t B, int64_t H, int64_t H_kv, int64_t S, int64_t D) {
  if (H_kv <= 0 || H <= 0 || H % H_kv != 0) return 0;
  int splits = 1;
  size_t delta_bytes = 0;
  return bwd_workspace_layout(B, H, H_kv, S, D, &splits, &delta_bytes);
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                 void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t S, int64_t D, int causal, float scale,
                 fa_dtype dtype, void* workspace, size_t workspace_bytes, void* stream) {
  return fa_bwd_marked(q, k, v, o, dout, lse, dq, dk, dv, B, H, S, D, causal, scale, dtype, workspace,
                       workspace_bytes, stream, nullptr);
}

fa_status fa_bwd_marked(const void* q, const void* k, const void* v, const void* o, const void* dout,
                        const float* lse, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t S, int64_t D,
                        int causal, float scale, fa_dtype dtype, void* workspace, size_t workspace_bytes,
                        void* stream, void* const* marks) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, B, H, H, S, D, causal, scale, dtype, workspace,
                  workspace_bytes, stream, marks);
}

fa_status fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                     void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t H_kv, int64_t S, int64_t D,
                     int causal, float scale, fa_dtype dtype, void* workspace, size_t workspace_bytes,
                     void* stream) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, S, D, causal, scale, dtype, workspace,
                  workspace_bytes, stream, nullptr);
}

fa_status fa_bwd_gqa_marked(const void* q, const void* k, const void* v, const void* o, const void* dout,
                            const float* lse, void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t H_kv,
                            int64_t S, int64_t D, int causal, float scale, fa_dtype dtype, void* workspace,
                            size_t workspace_bytes, void* stream, void* const* marks) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, B, H, H_kv, S, D, causal, scale, dtype, workspace,
                  workspace_bytes, stream, marks);
}

}  // extern "C"

namespace {

fa_status bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                   void* dq, void* dk, void* dv, int64_t B, int64_t H, int64_t H_kv, int64_t S, int64_t D,
                   int causal, float scale, fa_dtype dtype, void* workspace, size_t workspace_bytes,
                   void* stream, void* const* marks) {
  g_detail[0] = 0;
  fa_status st = check_common(B, H, S, D, scale, dtype);
  if (st != FA_OK) return st;
  if ((st = check_heads(H, H_kv))) return st;
  const int64_t BH = B * H;
  const int64_t BHkv = B * H_kv;
  if (BH == 0 || S == 0) return FA_OK;  // empty: nothing is read or written, pointers may be NULL
  if ((st = check_ptr(q, "q")) || (st = check_ptr(k, "k")) || (st = check_ptr(v, "v")) ||
      (st = check_ptr(o, "o")) || (st = check_ptr(dout, "dout")) || (st = check_ptr(lse, "lse")) ||
      (st = check_ptr(dq, "dq")) || (st = check_ptr(dk, "dk")) || (st = check_ptr(dv, "dv")))
    return st;
  int splits = 1;
  size_t delta_bytes = 0;
  const size_t need = bwd_workspace_layout(B, H, H_kv, S, D, &splits, &delta_bytes);
  if (!workspace) return fail(FA_ERR_WORKSPACE, "workspace is NULL (%zu bytes needed)", need);
  if (workspace_bytes < need)
    return fail(FA_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", workspace_bytes, need);
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(FA_ERR_ALIGNMENT, "workspace is not 256-byte aligned");
  const bool bf16 = dtype == FA_BF16;
  fa::BwdMaps maps;
  if ((st = encode_qkv_map(&maps.q128, q, bf16, D, S, BH, "q")) ||
      (st = encode_qkv_map(&maps.k128, k, bf16, D, S, BHkv, "k")) ||
      (st = encode_qkv_map(&maps.v128, v, bf16, D, S, BHkv, "v")) ||
      (st = encode_qkv_map(&maps.do128, dout, bf16, D, S, BH, "dout")) ||
      (st = encode_qkv_map(&maps.q64, q, bf16, D, S, BH, "q", 64)) ||
      (st = encode_qkv_map(&maps.k64, k, bf16, D, S, BHkv, "k", 64)) ||
      (st = encode_qkv_map(&maps.v64, v, bf16, D, S, BHkv, "v", 64)) ||
      (st = encode_qkv_map(&maps.do64, dout, bf16, D, S, BH, "dout", 64)))
    return st;
  fa::BwdParams p;
  p.o = o;
  p.dout = dout;
  p.lse = lse;
  p.delta = static_cast<float*>(workspace);
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.S = static_cast<int>(S);
  p.BH = static_cast<int>(BH);
  p.group = static_cast<int>(H / H_kv);
  p.kv_splits = splits;
  p.dkv_part = splits > 1 ? reinterpret_cast<float*>(static_cast<char*>(workspace) + delta_bytes) : nullptr;
  p.n_tiles = static_cast<int>((S + 127) / 128);
  p.n_partner = static_cast<int>((S + 63) / 64);
  p.causal = causal ? 1 : 0;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  p.err = fa::device_error_word();
  if (!p.err) return fail(FA_ERR_CUDA, "cannot resolve the device error word on the current device");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int Di = static_cast<int>(D);
  auto mark = [&](int i) -> fa_status {
    if (!marks || !marks[i]) return FA_OK;
    return from_cuda(cudaEventRecord(static_cast<cudaEvent_t>(marks[i]), s), "event record");
  };
  if ((st = mark(0))) return st;
  if ((st = from_cuda(fa::launch_bwd_preprocess(Di, bf16, p, s), "backward preprocess launch"))) return st;
  if ((st = mark(1))) return st;
  if ((st = from_cuda(fa::launch_bwd_dkdv(Di, bf16, maps, p, s), "backward dK/dV launch"))) return st;
  if (splits > 1 && (st = from_cuda(fa::launch_bwd_dkv_reduce(Di, bf16, p, s), "backward dK/dV reduce launch")))
    return st;
  if ((st = mark(2))) return st;
  if ((st = from_cuda(fa::launch_bwd_dq(Di, bf16, maps, p, s), "backward dQ launch"))) return st;
  return mark(3);
}

}  // namespace

extern "C" {

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
  // The same three kernels as fa_bwd, with the scratch array as the workspace.
  // The Delta kernel overwrites every row it uses, so nothing needs clearing.
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
    return fail(FA_ERR_TIMEOUT, "device pipeline wait timed out (code %d)", code);
  }
  return FA_OK;
}

}  // extern "C"
