// Shared definitions of the jagged flash attention kernels: tile sizes, the
// device work-list header, kernel parameter blocks and the host-side launch
// entry points implemented in the .cu files.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "errbits.cuh"

namespace jfa {

constexpr int kBM = 128;  // query rows per tile (one TMEM lane per row)
constexpr int kBN = 128;  // keys per tile
constexpr int kFwdRows = 256;  // query rows per forward work item (two tiles)

// Row statistics of the self-attention backward, {-LSE*log2e, -Delta} per
// query row (h, t) at row index si = h*T + t, in a blocked layout: every
// aligned group of 4 positions stores the 4 rows' -LSE*log2e (16 bytes),
// then their -Delta (16 bytes).  kStatCopies copies differ in where their
// groups start: copy k holds row si at position si + kStatPad - k, so a
// 128-row box starting at row s0 is 32 whole groups (1 KB, 32-byte aligned)
// of copy (s0 + kStatPad) % 4.  Positions of rows before 0 (a box of a
// batch shorter than one tile starts up to 127 rows early) hold zeros.
constexpr int kStatPad = 128;
constexpr int kStatCopies = 4;
__host__ __device__ __forceinline__ long long stat_pos(long long si, int k) {
  return si + kStatPad - k;
}
// float index of -LSE*log2e at position u (-Delta is 4 floats further)
__host__ __device__ __forceinline__ long long stat_float(long long u) {
  return (u >> 2) * 8 + (u & 3);
}
// floats per copy for rows [0, rows)
__host__ __device__ __forceinline__ long long stat_copy_floats(long long rows) {
  return ((2 * (rows + kStatPad + 4) + 63) / 64) * 64;
}

// Small header at the start of every scratch block, written by the
// scheduler kernel and read by the kernels that follow it on the stream.
struct WorkHeader {
  int n_items;  // number of work items in the list
  int T;        // offsets[B], total packed tokens
  int ticket;   // dynamic work counter of the persistent kernels
  int valid;    // 1 if offsets passed the device checks
  int pad[4];
};

// A work item: x = sequence b, y = (head << 16) | tile.
using Item = int2;

struct SchedParams {
  const int32_t* offsets;
  int B, H, Lq, max_len;
  int causal, broadcast, backward;
  int qrows;  // query rows per item when backward == 0 (forward and dQ pass: 256)
  Item* items;
  int capacity;
  WorkHeader* hdr;
  int* err;
};

struct FwdParams {
  const int32_t* offsets;
  int B, H, Lq;
  float scale_log2;  // scale * log2(e)
  __nv_bfloat16* out;
  float* lse;
  const Item* items;
  WorkHeader* hdr;
  int* err;
};

struct BwdParams {
  const int32_t* offsets;
  int B, H, Lq;
  float scale_log2;
  float scale;
  const float* lse;    // caller's LSE (natural log)
  const float* delta;  // broadcast: rowsum(dO * O), same layout as lse
  // Self-attention row statistics: kStatCopies copies of stat_stride floats
  // (layout at kStatPad above).
  const float* stat;
  long long stat_stride;
  float* dq_acc;       // fp32 accumulator: self [Tcap,H,D]; broadcast [shards,Lq,H,D]
  int dq_shards;       // broadcast only
  long long shard_stride;  // elements per shard
  __nv_bfloat16* dq;  // self-attention dQ pass: written directly
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  const Item* items;
  WorkHeader* hdr;
  int* err;
};

// Backward pre-pass: blocks [0, n_sched) build work lists, the others the
// row statistics.
struct PrepParams {
  const __nv_bfloat16* out;
  const __nv_bfloat16* dout;
  const int32_t* offsets;
  // self-attention: the row statistics as in BwdParams, from the caller's LSE
  const float* lse;
  float* stat;
  long long stat_stride;
  long long Tcap;  // B * max_len: rows of q, k, v, out, dout the caller provides
  // broadcast-Q: Delta [B, H, Lq] and the fp32 dQ accumulator to zero
  float* delta;
  float* dq_acc;
  long long dq_acc_elems_bcast;
  int B, H, D, Lq, broadcast;
  int n_sched;  // 1 or 2
  SchedParams sched[2];
};

struct FinParams {
  const float* dq_acc;
  __nv_bfloat16* dq;
  float scale;
  int H, D, Lq, broadcast, shards;
  long long shard_stride;
  const WorkHeader* hdr;
};

// Host-side launchers (return cudaGetLastError() after the launch).
cudaError_t launch_sched(const SchedParams& p, cudaStream_t s);
cudaError_t launch_fwd(int D, bool causal, bool bcast, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const FwdParams& p, int grid, cudaStream_t s);
cudaError_t launch_bwd(int D, bool causal, bool bcast, const CUtensorMap& tq,
                       const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                       const BwdParams& p, int grid, cudaStream_t s);
// tdk / tdv: the dK / dV outputs as maps like the inputs' (TMA stores).
cudaError_t launch_bwd_kv(int D, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& tdo, const CUtensorMap& tdk,
                          const CUtensorMap& tdv, const BwdParams& p, int grid, cudaStream_t s);
cudaError_t launch_bwd_q(int D, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, const CUtensorMap& tdo, const BwdParams& p,
                         int grid, cudaStream_t s);
cudaError_t launch_bwd_prep(const PrepParams& p, int sms, cudaStream_t s);
cudaError_t launch_finalize(const FinParams& p, int sms, cudaStream_t s);
cudaError_t launch_fill_empty(__nv_bfloat16* out, float* lse, long long rows, int D,
                              cudaStream_t s);
cudaError_t prepare_kernels(int device);

}  // namespace jfa
