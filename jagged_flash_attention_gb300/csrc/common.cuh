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

// Local (banded) attention: key j is admissible for query i, both counted
// from the start of their sequence, iff i - wl <= j <= i + wr.  kNoWindow
// leaves a side unbounded; causal masking is wl = kNoWindow, wr = 0.
// Lengths are below 2^23 (at most 65535 tiles), so i + kNoWindow cannot
// overflow.
constexpr int kNoWindow = 1 << 30;

// Key tiles [*j0, *j0 + *n) holding the admissible keys of query rows
// [qa, qb] of a sequence of L > 0 keys.
__host__ __device__ __forceinline__ void key_tiles(int qa, int qb, int L, int wl, int wr, int* j0,
                                                   int* n) {
  const int lo = qa - wl > 0 ? qa - wl : 0;
  const int hi = qb + wr < L - 1 ? qb + wr : L - 1;
  *j0 = lo / kBN;
  *n = hi / kBN - *j0 + 1;
}
// Query tiles [*t0, *t0 + *n) holding the queries (of L) that admit some key
// of rows [ka, kb].
__host__ __device__ __forceinline__ void query_tiles(int ka, int kb, int L, int wl, int wr, int* t0,
                                                     int* n) {
  const int lo = ka - wr > 0 ? ka - wr : 0;
  const int hi = kb + wl < L - 1 ? kb + wl : L - 1;
  *t0 = lo / kBM;
  *n = hi / kBM - *t0 + 1;
}

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
  int n_items;   // number of work items in the list
  int T;         // offsets[B], total packed tokens
  int ticket;    // dynamic work counter of the persistent kernels
  int valid;     // 1 if offsets passed the device checks
  int n_chunks;  // broadcast dQ pass: key-tile chunks per (head, query-tile pair)
  int pad[3];
};

// A work item: x = sequence b, y = (head << 16) | tile.
using Item = int2;

// Work item of the broadcast-Q dQ pass: head h and query-tile pair `pair`
// (hp = h | pair << 16), and a run of n key tiles of the concatenated
// key-tile stream of all sequences, starting at tile j of sequence b (b is
// non-empty; later tiles continue through the next non-empty sequences).
// The item's fp32 dQ partial goes to partial slot = its list index.
struct QbItem {
  int hp, b, j, n;
};

// Query rows per broadcast dQ-pass item (two 128-row tiles).
constexpr int kQbRows = 256;

// Position in the key-tile stream of the chunked broadcast kernels: key
// tile j of sequence b (which has nts tiles, keys [off0, off0 + L)).  The
// end offset of the next sequence is loaded when a sequence is entered, so
// that the step into the next sequence needs no global load on the spot.
struct Seg {
  int b, j, nts, off0, L;
  int nxt;  // offsets[b + 2] (or offsets[B] past the end)
};

__device__ __forceinline__ void seg_load(Seg& s, const int32_t* off, int B, int b, int j) {
  s.b = b;
  s.j = j;
  s.off0 = off[b];
  s.L = off[b + 1] - s.off0;
  s.nts = (s.L + kBN - 1) / kBN;
  s.nxt = b + 2 <= B ? off[b + 2] : s.off0 + s.L;
}

// Next key tile of the stream: the following tile of this sequence, else the
// first tile of the next non-empty sequence (never past sequence B - 1).
__device__ __forceinline__ void seg_next(Seg& s, const int32_t* off, int B) {
  if (++s.j < s.nts) return;
  const int b1 = s.b + 1, e1 = s.off0 + s.L;  // e1 = offsets[b1]
  if (b1 < B && s.nxt > e1) {
    s.b = b1;
    s.j = 0;
    s.off0 = e1;
    s.L = s.nxt - e1;
    s.nts = (s.L + kBN - 1) / kBN;
    s.nxt = b1 + 2 <= B ? off[b1 + 2] : s.nxt;
    return;
  }
  int b = b1;  // empty sequences follow
  while (b < B - 1 && off[b + 1] == off[b]) ++b;
  seg_load(s, off, B, b < B - 1 ? b : B - 1, 0);
}

struct SchedParams {
  const int32_t* offsets;
  int B, H, Lq, max_len;  // H: heads of the list (K/V heads for the dK/dV list)
  int causal, broadcast, backward;  // causal: any local mask (causal or a window)
  int qrows;  // query rows per item when backward == 0 (forward and dQ pass: 256)
  Item* items;
  int capacity;
  WorkHeader* hdr;
  int* err;
  int wl = kNoWindow, wr = kNoWindow;  // the local mask, for the cost order
  // Block-sparse forward: the lists the forward will follow, checked here
  // (nullptr: none).
  const int32_t* blocks = nullptr;
  const int32_t* counts = nullptr;
  int nqb = 0, kcap = 0;
  // their check, by list_check_kernel: one result per block (1: valid)
  int* check = nullptr;
  int n_check = 0;
  int kpair = 1;  // backward: key blocks per item (2: pairs of CTAs)
};

// Every parameter block below carries the GQA group G (query heads per K/V
// head: query head h reads K/V head h / G) and the local mask (wl, wr); the
// host sets them on every path.
struct FwdParams {
  const int32_t* offsets;
  int B, H, Lq;
  int G, wl, wr;
  float scale_log2;  // scale * log2(e)
  __nv_bfloat16* out;
  float* lse;
  const Item* items;
  WorkHeader* hdr;
  int* err;
  // Streamed broadcast forward (fwd_bs.cu): key-tile chunks, the key-tile
  // prefix per sequence, and the partials of split sequences ([items][2]
  // pieces x 128 rows: O / l fp32 [.., D] and the base-2 LSE).
  const QbItem* qb_items;
  const int* kt_off;
  float* part_o;
  float* part_lse;
  // Block-sparse forward: key-tile lists [B][H][nqb][kcap] and their counts.
  const int32_t* blocks;
  const int32_t* counts;
  int nqb, kcap;
};

struct BwdParams {
  const int32_t* offsets;
  int B, H, Lq;
  int Hkv, G, wl, wr;  // K/V heads (dK, dV are [T, Hkv, D]), group, local mask
  float scale_log2;
  float scale;
  const float* lse;    // caller's LSE (natural log)
  // Row statistics {-LSE*log2e, -Delta} in the blocked layout of stat_float:
  // self-attention, kStatCopies copies of stat_stride floats (layout at
  // kStatPad above); broadcast, one copy over [B, H, Lq rounded up to 128]
  // with padding rows {-inf, 0}.
  const float* stat;
  long long stat_stride;
  float* dq_part;      // broadcast dQ pass: fp32 partial of each item
  __nv_bfloat16* dq;  // self-attention dQ pass: written directly
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  const Item* items;
  const QbItem* qb_items;  // broadcast dQ pass
  WorkHeader* hdr;
  int* err;
};

// Work list of the broadcast-Q dQ pass (built by one block of the pre-pass):
// the key-tile stream of every (head, pair) cut into n equal chunks, n =
// min(chunk_cap, ceil(tiles / 4)), where tiles = sum_b ceil(L_b / 128).
struct QbSchedParams {
  const int32_t* offsets;
  int B, H, Lq, max_len;
  int chunk_cap;  // chunks per (head, pair) at most
  int* kt_off;    // scratch int[B + 1]: key tiles before sequence b
  QbItem* items;
  int capacity;   // chunk_cap * H * pairs
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
  int B, H, D, Lq, broadcast;
  // Work lists: n_sched = 2; block 0 builds sched[0]; block 1 builds
  // sched[1] (self-attention) or the broadcast dQ-pass list qb.
  int n_sched;
  SchedParams sched[2];
  QbSchedParams qb;
  int qb_only;  // broadcast one-pass backward: block 0 builds the dQ-pass list alone
};

// Broadcast dQ: dq[l, h, :] = bf16(scale * sum over the chunks of the
// partials of (h, pair = l / 256)), chunks summed in a fixed order.
struct FinParams {
  const float* part;  // [n_items][2][128][D] fp32, list order of QbSchedParams
  __nv_bfloat16* dq;
  float scale;
  int H, D, Lq;
  const WorkHeader* hdr;  // header of the dQ-pass list (n_chunks, valid)
};

// Block-sparse attention, stage 1 (sparse.cu): K-block means, then per
// (sequence, query head, 256-row Q block) the top-k of its sequence's
// 128-key K blocks by the dot product of the two means.  Lists: blocks
// [B][H][nqb][kcap] (ascending, -1 after counts), counts [B][H][nqb].
constexpr int kSparseMaxKBlocks = 2048;  // kcap limit: max_len <= 262144
struct SparseParams {
  const __nv_bfloat16* q;  // [T, H, D]
  const __nv_bfloat16* k;  // [T, Hkv, D]
  const int32_t* offsets;
  int B, H, Hkv, G, D, max_len, permille;
  int Lq, broadcast;  // broadcast-Q: the Q blocks are the dense Q's (q is [Lq, H, D])
  int nqb, kcap;  // ceil(max_len / 256) (broadcast: ceil(Lq / 256)), ceil(max_len / 128)
  int wl, wr;     // local mask [i - wl, i + wr] (kNoWindow: unbounded side)
  float* kbar;     // scratch fp32 [B][Hkv][kcap][D]: K-block means
  float* qsum;     // scratch fp32 [B][H][2 nqb][D]: sums of 128-row Q halves (broadcast: [1][H][2 nqb][D])
  int32_t* blocks;
  int32_t* counts;
  int* err;
};

// Host-side launchers (return cudaGetLastError() after the launch).
cudaError_t launch_sched(const SchedParams& p, cudaStream_t s);
// Block lists of the sparse forward, checked before the scheduler reads the
// results: list_check_blocks(p) result slots (p.n_check of them).
int list_check_blocks(const SchedParams& p);
cudaError_t launch_list_check(const SchedParams& p, cudaStream_t s);
// causal: any local mask (the kernels read wl, wr from the parameters).
// sparse: the block-sparse forward (self-attention, no mask; p.blocks).
cudaError_t launch_fwd(int D, bool causal, bool bcast, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const FwdParams& p, int grid, cudaStream_t s,
                       bool sparse = false);
// tdk / tdv: the dK / dV outputs as maps like the inputs' (TMA stores).
// With tq_h and tdo_h (maps of Q and dO with 64-row boxes), the pair
// variant: clusters of two CTAs over a list of key-block pairs (D = 128,
// no local mask).
cudaError_t launch_bwd_kv(int D, bool causal, bool bcast, const CUtensorMap& tq,
                          const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                          const CUtensorMap& tdk, const CUtensorMap& tdv, const BwdParams& p,
                          int grid, cudaStream_t s, const CUtensorMap* tq_h = nullptr,
                          const CUtensorMap* tdo_h = nullptr);
// Broadcast-Q forward for a short dense Q (q_len <= 128), streamed over
// key-tile chunks (fwd_bs.cu), and the merge of split sequences.
bool fwd_bs_supported(int Lq);
// q_len <= 64: the spread layout (the Q map's box must then be 16 rows high).
bool fwd_bs_spread(int Lq);
cudaError_t launch_fwd_bs(int D, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const FwdParams& p, int grid, cudaStream_t s);
cudaError_t launch_fwd_combine(int D, const FwdParams& p, int sms, cudaStream_t s);
// Broadcast-Q backward in one pass for a short dense Q (bwd_bs.cu): dK, dV
// and the dQ partials of the items of the dQ-pass list.
bool bwd_bs_supported(int D, int Lq);
cudaError_t launch_bwd_bs(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const BwdParams& p, int grid, cudaStream_t s);
// Broadcast-Q dQ pass (tdo: the 4-D [B, Lq, H, D] map).
cudaError_t launch_bwd_qb(int D, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& tdo, const BwdParams& p,
                          int grid, cudaStream_t s);
cudaError_t launch_bwd_q(int D, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, const CUtensorMap& tdo, const BwdParams& p,
                         int grid, cudaStream_t s);
cudaError_t launch_bwd_prep(const PrepParams& p, int sms, cudaStream_t s);
cudaError_t launch_qb_sched(const QbSchedParams& p, cudaStream_t s);
// Copies a work list out (4 ints per item) with its counts (list inspection).
cudaError_t launch_export_list(const WorkHeader* hdr, const void* items, int qb, int32_t* out,
                               int capacity, int32_t* count, cudaStream_t s);
cudaError_t launch_finalize(const FinParams& p, int sms, cudaStream_t s);
cudaError_t launch_sparse_pool(const SparseParams& p, cudaStream_t s);
cudaError_t launch_sparse_select(const SparseParams& p, cudaStream_t s);
cudaError_t launch_fill_empty(__nv_bfloat16* out, float* lse, long long rows, int D,
                              cudaStream_t s);
cudaError_t prepare_kernels(int device);

}  // namespace jfa
