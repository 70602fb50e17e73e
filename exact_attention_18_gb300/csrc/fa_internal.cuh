// Internal declarations shared by the host entry points and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

constexpr int kBlockM = 128;  // query rows per tile (= TMEM lanes)
constexpr int kBlockN = 128;  // key rows per tile
constexpr int kNoWindow = 1 << 30;  // an unlimited window side (larger than any sequence)

// Two layouts.  Fixed length (cu_seqlens == nullptr): [B*H, S, D] tensors,
// row r of head bh at element (bh*S + r)*D, L at bh*S + r, tensor maps
// {D, S, heads}.  Packed batch (cu_seqlens != nullptr): [T, H, D] tensors
// (token-major), sample b = tokens cu[b] .. cu[b+1]-1, its row r is token
// cu[b] + r; L is [H, T]; tensor maps {D, heads, T}; S is then the largest
// sample length and blockIdx.x = b*H + h.
struct FwdParams {
  void* o;             // [BH, S, D] or [T, H, D] output
  float* lse;          // [BH, S] or [H, T] natural-log logsumexp
  int S;               // sequence length (packed batch: max_seqlen)
  const int* cu_seqlens;  // packed batch: [B + 1] token offsets in device memory; else nullptr
  int heads;           // H (query heads per batch entry)
  int total;           // packed batch: T tokens
  int n_m_tiles;       // CTAs per (b, h): ceil(S / fwd_rows_per_cta(D))
  int causal;          // nonzero: key j visible to query i iff j <= i
  int win_left;        // general kernels: key j visible to query i iff i - win_left <= j <= i + win_right
  int win_right;       // (kNoWindow = unlimited; causal sets win_right = 0)
  int group;           // query heads per K/V head: query head bh reads K/V head bh / group
  int kv_chunk;        // general kernels, split-KV: keys per shard (a multiple of 128; 0 = no split);
                       // shard z = blockIdx.z covers keys [z*kv_chunk, (z+1)*kv_chunk)
  float* o_part;       // split-KV: fp32 O of each shard, [shards][B*H*S][D] (else nullptr)
  float* lse_part;     // split-KV: fp32 natural-log L of each shard, [shards][B*H*S]
  float scale_log2;    // scale * log2(e): scores enter exp2 in base 2
  int* err;            // device error word (set when a pipeline wait times out)
  unsigned long long wait_ns;  // limit of each pipeline wait (fa_set_wait_limit_ns)
};

struct BwdParams {
  const void* o;       // [BH, S, D] (or [T, H, D]) forward output (BH counts query heads)
  const void* dout;    // [BH, S, D] loss gradient w.r.t. O
  const float* lse;    // [BH, S] natural-log logsumexp from the forward
  float* delta;        // [BH, S] workspace: rowsum(dO o O)
  void* dq;            // [BH, S, D]
  void* dk;            // [BH / group, S, D]
  void* dv;            // [BH / group, S, D]
  int S;               // sequence length (packed batch: max_seqlen)
  const int* cu_seqlens;  // packed batch: [B + 1] token offsets in device memory; else nullptr
  int heads;           // H
  int total;           // packed batch: T tokens
  int BH;              // query heads B*H
  int group;           // query heads per K/V head (H / H_kv); K/V head of query head bh is bh / group
  int kv_splits;       // dK/dV pass: CTAs sharing a (K/V head, key tile), each over group / kv_splits heads
  float* dkv_part;     // kv_splits > 1: fp32 partial sums [kv_splits][K/V rows][2 D] (dV | scale*dK),
                       // K/V rows in dK's own row order (B*H_kv*S, or T*H_kv packed)
  int n_tiles;         // ceil(S / 128): own tiles per (b, h)
  int causal;
  int win_left;        // general kernels: window as in FwdParams
  int win_right;
  float scale;         // softmax scale (dQ, dK factor)
  float scale_log2;    // scale * log2(e)
  int* err;            // device error word
  unsigned long long wait_ns;  // limit of each pipeline wait (fa_set_wait_limit_ns)
};

// Tensor maps of the backward's four inputs, each viewed as 3-D {D, S, heads}
// (B*H heads for Q and dO, B*H_kv for K and V):
// 128-row boxes for a CTA's resident tiles, 64-row boxes for streamed blocks.
struct BwdMaps {
  CUtensorMap q128, k128, v128, do128;
  CUtensorMap q64, k64, v64, do64;
};

// Query rows one forward CTA covers for head dimension D.
int fwd_rows_per_cta(int D);

// Launchers (one per kernel family); they dispatch on D and dtype, and take
// the general instantiation (packed batches, windows) when `general` is set;
// the fixed-length full/causal calls run the specialised one.
// launch_fwd4: the forward for D <= 64 (the persistent two-pipeline kernel,
// launch_fwd4p, for fixed-length calls; the four-tile kernel for the general
// ones); launch_fwd: any D (passes D <= 64 on to launch_fwd4).
cudaError_t launch_fwd4(int D, bool bf16, bool general, const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv, const FwdParams& p, int BH, cudaStream_t stream);
cudaError_t launch_fwd4p(int D, bool bf16, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const FwdParams& p, int BH, cudaStream_t stream);
cudaError_t launch_fwd(int D, bool bf16, bool general, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const FwdParams& p, int BH, cudaStream_t stream);

// rows: query rows (B*H*S, or T*H packed).
// Split-KV merge: O = sum_s exp(L_s - L) O_s, L = ln sum_s exp(L_s), per row.
cudaError_t launch_merge_lse(int D, bool bf16, const float* o_part, const float* lse_part, int shards, int64_t rows,
                             void* o, float* lse, cudaStream_t stream);

cudaError_t launch_bwd_preprocess(int D, bool bf16, const BwdParams& p, int64_t rows, cudaStream_t stream);
// dependent: launch as a programmatic dependent launch of the kernel just
// before it on `stream` (a backward kernel of the same call): its CTAs may
// start while that kernel runs, and it waits for that kernel's grid before it
// reads Delta.  Only the kernel that computes Delta (the Delta kernel, or the
// persistent dQ pass) runs before them otherwise; the dK/dV pass (and its
// partial-sum reduction) writes nothing the dQ pass reads.
cudaError_t launch_bwd_dkdv(int D, bool bf16, bool general, const BwdMaps& maps, const BwdParams& p,
                            cudaStream_t stream, bool dependent);
cudaError_t launch_bwd_dq(int D, bool bf16, bool general, const BwdMaps& maps, const BwdParams& p,
                          cudaStream_t stream, bool dependent);
// True when launch_bwd_dq's kernel computes Delta itself and writes it to p.delta
// (the persistent dQ kernel): the backward then skips the Delta kernel and runs
// the dQ pass before the dK/dV pass, which reads that Delta.
bool bwd_dq_computes_delta(int D, bool general);
// Sums the kv_splits partial dK/dV rows and writes dK, dV (only when kv_splits > 1);
// rows: K/V rows (B*H_kv*S, or T*H_kv packed).
cudaError_t launch_bwd_dkv_reduce(int D, bool bf16, const BwdParams& p, int64_t rows, cudaStream_t stream);

// CTAs per (K/V head, key tile) in the dK/dV pass: the smallest divisor of
// `group` that gives at least two CTAs per SM of a 152-SM GPU (1 when the
// heads alone do, or for ordinary multi-head attention).
int bwd_kv_splits(int64_t BHkv, int64_t n_tiles, int group);

// Address of this process's device error word on the current device.
int* device_error_word();

// Limit the kernels launched next give each pipeline wait (nanoseconds).
unsigned long long wait_limit_ns();

// Bytes per swizzled shared-memory row for head dimension D (16-bit elements):
// 32 for D = 16, 64 for D = 32, 128 for D >= 64 (D = 128 uses two column chunks).
inline int row_bytes_for(int D) { return D * 2 < 128 ? D * 2 : 128; }

}  // namespace fa
