// Block-sparse attention, stage 1: block scores and top-k block selection.
//
// "Optimizing Jagged Flash Attention with TLX" (pytorch.org), section 3,
// "Block-sparse attention": a cheap scoring step average-pools each Q block
// and each K block and keeps, per Q block, the top-k most relevant K/V
// blocks; the attention (stage 2, fwd.cu with the block list) then runs over
// the selected blocks only.  Blocks here: K blocks are the 128-key tiles of a
// sequence, Q blocks its 256-row forward work items, so that the two query
// tiles of an item share one list.  k = max(1, ceil(permille * n / 1000)) of
// the sequence's n K blocks; ties go to the lower block index; lists are
// stored in ascending order.
//
// Two kernels:
//   sparse_pool_kernel     K-block and Q-block means (fp32 scratch), reading
//                          K and Q once in 16-byte chunks
//   sparse_select_kernel   per (Q block, query head, sequence): the dot
//                          products of the Q-block mean with the sequence's
//                          K-block means, the rank of every score, the
//                          selected blocks in ascending order.  With a local
//                          mask (causal or a window) only the K blocks that
//                          hold an admissible key of some row of the Q block
//                          are candidates, and k counts from them.
#include "common.cuh"
#include "ptx.cuh"

namespace jfa {
namespace {

constexpr int kPoolThreads = 256;
constexpr int kSelThreads = 256;

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

// Rows [off0, off0 + L) of sequence b lie inside [0, offsets[B]) and L <=
// max_len; otherwise the device error word gets kErrBadOffsets and the
// sequence is skipped, so that no read leaves the caller's buffers.
__device__ __forceinline__ bool seq_ok(const SparseParams& p, int off0, int L) {
  const bool ok = p.offsets[0] == 0 && off0 >= 0 && L >= 0 && L <= p.max_len &&
                  off0 + L <= p.offsets[p.B];
  if (!ok && threadIdx.x == 0) atomicOr(p.err, kErrBadOffsets);
  return ok;
}

// Mean of the valid rows of one row block of a sequence, for every head of
// a [T, Hx, D] tensor: out[h * out_stride + d].  A row of all heads (Hx * D
// bf16, contiguous) is read as 16-byte chunks: with fewer chunks than
// threads, thread t takes chunk t % cpr of rows t / cpr, + groups, ... and
// the row groups are added in shared memory (at most kPoolThreads * 8
// floats); otherwise every thread owns whole chunks.
__device__ void pool_rows(const __nv_bfloat16* x, int Hx, int D, long long row0, int n,
                          float* out, long long out_stride, float* part) {
  const int W = Hx * D;     // elements per row
  const int cpr = W / 8;    // 16-byte chunks per row
  const int t = threadIdx.x;
  const long long base = row0 * W;
  auto load_add = [&](float (&acc)[8], long long e) {
    const uint4 u = *reinterpret_cast<const uint4*>(x + e);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
      acc[2 * k] += f.x;
      acc[2 * k + 1] += f.y;
    }
  };
  const float inv = 1.f / n;
  if (cpr >= kPoolThreads) {
    for (int c = t; c < cpr; c += kPoolThreads) {
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
      for (int r = 0; r < n; ++r) load_add(acc, base + static_cast<long long>(r) * W + c * 8);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int col = c * 8 + k;
        out[(col / D) * out_stride + col % D] = acc[k] * inv;
      }
    }
    return;
  }
  const int groups = kPoolThreads / cpr, c = t % cpr, g = t / cpr;
  if (g < groups) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
    for (int r = g; r < n; r += groups)
      load_add(acc, base + static_cast<long long>(r) * W + c * 8);
#pragma unroll
    for (int k = 0; k < 8; ++k) part[g * W + c * 8 + k] = acc[k];
  }
  __syncthreads();
  for (int col = t; col < W; col += kPoolThreads) {
    float s = 0.f;
    for (int q = 0; q < groups; ++q) s += part[q * W + col];
    out[(col / D) * out_stride + col % D] = s * inv;
  }
}

// One CTA per (block j, sequence b, tensor z): z = 0, K block j (128 keys)
// for every K/V head into kbar [B][Hkv][kcap][D]; z = 1, Q block j (256
// rows) for every query head into qbar [B][H][nqb][D] (broadcast-Q: the
// dense Q's block j, once, into qbar [H][nqb][D]).
__global__ void __launch_bounds__(kPoolThreads) sparse_pool_kernel(SparseParams p) {
  __shared__ float part[kPoolThreads * 8];
  const int j = blockIdx.x, b = blockIdx.y;
  const int off0 = p.offsets[b];
  const int L = p.offsets[b + 1] - off0;
  if (!seq_ok(p, off0, L)) return;
  if (blockIdx.z == 0) {
    const int r0 = j * kBN;
    if (j >= p.kcap || r0 >= L) return;
    pool_rows(p.k, p.Hkv, p.D, off0 + r0, min(kBN, L - r0),
              p.kbar + (static_cast<long long>(b) * p.Hkv * p.kcap + j) * p.D,
              static_cast<long long>(p.kcap) * p.D, part);
  } else if (p.broadcast) {  // the dense Q's blocks, once (by the CTAs of sequence 0)
    const int r0 = j * kFwdRows;
    if (b != 0 || j >= p.nqb) return;
    pool_rows(p.q, p.H, p.D, r0, min(kFwdRows, p.Lq - r0), p.qbar + static_cast<long long>(j) * p.D,
              static_cast<long long>(p.nqb) * p.D, part);
  } else {
    const int r0 = j * kFwdRows;
    if (j >= p.nqb || r0 >= L) return;
    pool_rows(p.q, p.H, p.D, off0 + r0, min(kFwdRows, L - r0),
              p.qbar + (static_cast<long long>(b) * p.H * p.nqb + j) * p.D,
              static_cast<long long>(p.nqb) * p.D, part);
  }
}

// One CTA per (Q block i, query head h, sequence b).
__global__ void __launch_bounds__(kSelThreads) sparse_select_kernel(SparseParams p) {
  __shared__ float score[kSparseMaxKBlocks];
  __shared__ int flag[kSparseMaxKBlocks];
  __shared__ int warp_sum[kSelThreads / 32];
  const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int off0 = p.offsets[b];
  const int L = p.offsets[b + 1] - off0;
  const long long row = (static_cast<long long>(b) * p.H + h) * p.nqb + i;
  int32_t* list = p.blocks + row * p.kcap;
  const int q0 = i * kFwdRows;
  // no such Q block, a sequence without keys (broadcast), or bad offsets: an empty list
  if (!seq_ok(p, off0, L) || (p.broadcast ? L == 0 : q0 >= L)) {
    for (int c = t; c < p.kcap; c += kSelThreads) list[c] = -1;
    if (t == 0) p.counts[row] = 0;
    return;
  }
  const int D = p.D;
  const int nk = cdiv(L, kBN);
  const int hk = h / p.G;
  // Candidates: K blocks [jlo, jhi) holding keys of [q0 - wl, q_last + wr]
  // (all of them without a local mask; kNoWindow keeps the sums in range).
  const int q_last = (p.broadcast ? min(p.Lq, q0 + kFwdRows) : min(L, q0 + kFwdRows)) - 1;
  const int jlo = max(0, q0 - p.wl) / kBN;
  const int jhi = min(L - 1, q_last + p.wr) / kBN + 1;
  // the Q block's mean (row = (b * H + h) * nqb + i; broadcast: one dense Q for all b)
  const float* qm = p.qbar + (p.broadcast ? static_cast<long long>(h) * p.nqb + i : row) * D;
  // Scores: one warp per K block, lanes over the head dimension.
  const float* kb = p.kbar + (static_cast<long long>(b) * p.Hkv + hk) * p.kcap * D;
  for (int j = jlo + warp; j < jhi; j += kSelThreads / 32) {
    float s = 0.f;
    for (int d = lane; d < D; d += 32) s += qm[d] * kb[static_cast<long long>(j) * D + d];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) score[j] = s;
  }
  __syncthreads();
  // Rank of every score (larger first, ties to the lower index); the k best
  // are selected.
  const int nc = jhi - jlo;
  const int k = min(nc, max(1, (p.permille * nc + 999) / 1000));
  for (int j = t; j < nk; j += kSelThreads) {
    int f = 0;
    if (j >= jlo && j < jhi) {
      const float sj = score[j];
      int rank = 0;
      for (int m = jlo; m < jhi; ++m) {
        const float sm = score[m];
        rank += (sm > sj || (sm == sj && m < j)) ? 1 : 0;
      }
      f = rank < k ? 1 : 0;
    }
    flag[j] = f;
  }
  __syncthreads();
  // Selected blocks in ascending order: a block-wide prefix count per chunk
  // of kSelThreads indices.
  int base = 0;
  for (int c0 = 0; c0 < nk; c0 += kSelThreads) {
    const int j = c0 + t;
    const int f = j < nk ? flag[j] : 0;
    const unsigned bal = __ballot_sync(0xffffffffu, f);
    if (lane == 0) warp_sum[warp] = __popc(bal);
    __syncthreads();
    int before = base;
    for (int w = 0; w < warp; ++w) before += warp_sum[w];
    before += __popc(bal & ((1u << lane) - 1u));
    if (f) list[before] = j;
    int tot = 0;
    for (int w = 0; w < kSelThreads / 32; ++w) tot += warp_sum[w];
    base += tot;
    __syncthreads();
  }
  for (int c = k + t; c < p.kcap; c += kSelThreads) list[c] = -1;
  if (t == 0) p.counts[row] = k;
}

}  // namespace

cudaError_t launch_sparse_pool(const SparseParams& p, cudaStream_t s) {
  sparse_pool_kernel<<<dim3(max(p.kcap, p.nqb), p.B, 2), kPoolThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_sparse_select(const SparseParams& p, cudaStream_t s) {
  sparse_select_kernel<<<dim3(p.nqb, p.H, p.B), kSelThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace jfa
