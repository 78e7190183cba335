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
//   sparse_pool_kernel     one CTA per 128-row unit of K (the K block's mean)
//                          or of Q (the sum of its rows; a Q block's mean is
//                          formed from its two halves when it is scored), all
//                          units the same size, each row of all heads read
//                          once in 16-byte chunks with several loads of a
//                          thread in flight
//   sparse_select_kernel   per (Q block, query head, sequence): the dot
//                          products of the Q-block mean with the sequence's
//                          K-block means, the rank of every score, the
//                          selected blocks in ascending order; one warp per
//                          list when a sequence has at most 128 K blocks, one
//                          CTA per list otherwise.  With a local mask (causal
//                          or a window) only the K blocks that hold an
//                          admissible key of some row of the Q block are
//                          candidates, and k counts from them.
#include "common.cuh"
#include "ptx.cuh"

namespace jfa {
namespace {

constexpr int kPoolBatch = 8;  // row loads a pooling thread issues before adding them
constexpr int kSelThreads = 256;
constexpr int kSelWarps = kSelThreads / 32;
constexpr int kUnit = 128;  // rows of a pooling unit (a K block, half a Q block)

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

// Rows [off0, off0 + L) of sequence b lie inside [0, offsets[B]) and L <=
// max_len; otherwise the device error word gets kErrBadOffsets (reported by
// the calling thread when `report`) and the sequence is skipped, so that no
// read leaves the caller's buffers.
__device__ __forceinline__ bool seq_ok(const SparseParams& p, int off0, int L, bool report) {
  const bool ok = p.offsets[0] == 0 && off0 >= 0 && L >= 0 && L <= p.max_len &&
                  off0 + L <= p.offsets[p.B];
  if (!ok && report) atomicOr(p.err, kErrBadOffsets);
  return ok;
}

// scale * (sum of rows [row0, row0 + n)), n <= kUnit, for every head of a
// [T, Hx, D] tensor: out[h * out_stride + d].  A row of all heads (Hx * D
// bf16, contiguous) is read as 16-byte chunks: with fewer chunks than
// threads, thread t takes chunk t % cpr of rows t / cpr, + groups, ... and
// the row groups are added in shared memory (at most NT * 8 floats);
// otherwise every thread owns whole chunks.  A thread issues kPoolBatch row
// loads before it adds them.
template <int NT>
__device__ void pool_rows(const __nv_bfloat16* x, int Hx, int D, long long row0, int n,
                          float scale, float* out, long long out_stride, float* part) {
  const int W = Hx * D;     // elements per row
  const int cpr = W / 8;    // 16-byte chunks per row
  const int t = threadIdx.x;
  const long long base = row0 * W;
  auto add = [](float (&acc)[8], const uint4& u) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
      acc[2 * k] += f.x;
      acc[2 * k + 1] += f.y;
    }
  };
  // rows first, first + step, ... below n, of chunk column c
  auto sum_rows = [&](float (&acc)[8], int c, int first, int step) {
    for (int r0 = first; r0 < n; r0 += step * kPoolBatch) {
      uint4 u[kPoolBatch];
#pragma unroll
      for (int q = 0; q < kPoolBatch; ++q) {
        const int r = r0 + q * step;
        u[q] = r < n ? *reinterpret_cast<const uint4*>(x + base + static_cast<long long>(r) * W + c * 8)
                     : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int q = 0; q < kPoolBatch; ++q) add(acc, u[q]);
    }
  };
  if (cpr >= NT) {
    for (int c = t; c < cpr; c += NT) {
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      sum_rows(acc, c, 0, 1);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int col = c * 8 + k;
        out[(col / D) * out_stride + col % D] = acc[k] * scale;
      }
    }
    return;
  }
  const int groups = NT / cpr, c = t % cpr, g = t / cpr;
  if (g < groups) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    sum_rows(acc, c, g, groups);
#pragma unroll
    for (int k = 0; k < 8; ++k) part[g * W + c * 8 + k] = acc[k];
  }
  __syncthreads();
  for (int col = t; col < W; col += NT) {
    float s = 0.f;
    for (int q = 0; q < groups; ++q) s += part[q * W + col];
    out[(col / D) * out_stride + col % D] = s * scale;
  }
}

// One CTA per (128-row unit j, sequence b, tensor z): z = 0, K block j, its
// mean for every K/V head into kbar [B][Hkv][kcap][D]; z = 1, query rows
// [128 j, 128 j + 128) of the sequence, their sum for every query head into
// qsum [B][H][2 nqb][D] (broadcast-Q: rows of the dense Q, once, by the CTAs
// of sequence 0, into qsum [H][2 nqb][D]).
// NT threads: 512 for rows of at most 1024 elements (each thread then adds
// 32 rows of a unit), 256 for wider rows (measured: 66 -> 59 us on H D = 1024;
// 204 -> 223 us on H D = 2048 with 512).
template <int NT>
__global__ void __launch_bounds__(NT) sparse_pool_kernel(SparseParams p) {
  __shared__ float part[NT * 8];
  const int j = blockIdx.x, b = blockIdx.y;
  const int off0 = p.offsets[b];
  const int L = p.offsets[b + 1] - off0;
  if (!seq_ok(p, off0, L, threadIdx.x == 0)) return;
  const int nh = 2 * p.nqb;  // 128-row halves of the Q blocks
  const int r0 = j * kUnit;
  if (blockIdx.z == 0) {
    if (j >= p.kcap || r0 >= L) return;
    const int n = min(kUnit, L - r0);
    pool_rows<NT>(p.k, p.Hkv, p.D, off0 + r0, n, 1.f / n,
              p.kbar + (static_cast<long long>(b) * p.Hkv * p.kcap + j) * p.D,
              static_cast<long long>(p.kcap) * p.D, part);
  } else if (p.broadcast) {
    if (b != 0 || j >= nh || r0 >= p.Lq) return;
    pool_rows<NT>(p.q, p.H, p.D, r0, min(kUnit, p.Lq - r0), 1.f,
              p.qsum + static_cast<long long>(j) * p.D, static_cast<long long>(nh) * p.D, part);
  } else {
    if (j >= nh || r0 >= L) return;
    pool_rows<NT>(p.q, p.H, p.D, off0 + r0, min(kUnit, L - r0), 1.f,
              p.qsum + (static_cast<long long>(b) * p.H * nh + j) * p.D,
              static_cast<long long>(nh) * p.D, part);
  }
}

// What both selection kernels need about list (b, h, i).
struct ListCtx {
  long long row;  // (b * H + h) * nqb + i
  int L, nk;      // the sequence's keys and K blocks
  int jlo, jhi;   // candidate K blocks [jlo, jhi)
  int nq;         // rows of the Q block
  bool has1;      // the Q block's second 128-row half exists
  bool empty;     // nothing to select: an empty list
};

// Candidates: K blocks [jlo, jhi) holding keys of [q0 - wl, q_last + wr]
// (all of them without a local mask; kNoWindow keeps the sums in range).
__device__ __forceinline__ ListCtx list_ctx(const SparseParams& p, int b, int h, int i,
                                            bool report) {
  ListCtx x;
  x.row = (static_cast<long long>(b) * p.H + h) * p.nqb + i;
  const int off0 = p.offsets[b];
  x.L = p.offsets[b + 1] - off0;
  const int q0 = i * kFwdRows;
  // no such Q block, a sequence without keys (broadcast), or bad offsets
  x.empty = !seq_ok(p, off0, x.L, report) || (p.broadcast ? x.L == 0 : q0 >= x.L);
  if (x.empty) return x;
  const int rows = p.broadcast ? p.Lq : x.L;
  x.nq = min(kFwdRows, rows - q0);
  x.has1 = q0 + kUnit < rows;
  x.nk = cdiv(x.L, kBN);
  const int q_last = q0 + x.nq - 1;
  x.jlo = max(0, q0 - p.wl) / kBN;
  x.jhi = min(x.L - 1, q_last + p.wr) / kBN + 1;
  return x;
}

// The first of the two 128-row half sums of the Q block of list (b, h, i)
// (the second follows it, D floats later, when it exists).
__device__ __forceinline__ const float* q_halves(const SparseParams& p, int b, int h, int i) {
  const long long hrow = (p.broadcast ? 0LL : static_cast<long long>(b) * p.H) + h;
  return p.qsum + (hrow * (2 * p.nqb) + 2 * i) * p.D;
}

__device__ __forceinline__ int k_count(int permille, int n) {
  return min(n, max(1, (permille * n + 999) / 1000));
}

// One warp per list, for sequences of at most 32 PER K blocks (kcap <= 32
// PER): lane d + 32 t holds the Q-block mean's column d + 32 t; the scores
// of 8 candidates at a time are loaded together (lanes over the head
// dimension, every load of the batch in flight at once) and reduced across
// the warp, candidate c's ending in lane c % 32 (slot c / 32); ranks by
// shuffles, the selected blocks compacted by a ballot per 32 candidates.
template <int PER>
__global__ void __launch_bounds__(kSelThreads, 4) sparse_select_warp_kernel(SparseParams p) {
  constexpr int kBatch = 8;
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const long long r = static_cast<long long>(blockIdx.x) * kSelWarps + (threadIdx.x >> 5);
  if (r >= static_cast<long long>(p.B) * p.H * p.nqb) return;
  const int i = static_cast<int>(r % p.nqb);
  const int h = static_cast<int>((r / p.nqb) % p.H);
  const int b = static_cast<int>(r / (static_cast<long long>(p.nqb) * p.H));
  const ListCtx x = list_ctx(p, b, h, i, lane == 0);
  int32_t* list = p.blocks + x.row * p.kcap;
  if (x.empty) {
    for (int c = lane; c < p.kcap; c += 32) list[c] = -1;
    if (lane == 0) p.counts[x.row] = 0;
    return;
  }
  const int D = p.D, nt = D / 32;
  const float* qs = q_halves(p, b, h, i);
  const float inv = 1.f / x.nq;
  float qm[4];
#pragma unroll
  for (int t = 0; t < 4; ++t)
    qm[t] = t < nt ? (qs[lane + 32 * t] + (x.has1 ? qs[D + lane + 32 * t] : 0.f)) * inv : 0.f;
  const float* kb = p.kbar + ((static_cast<long long>(b) * p.Hkv + h / p.G) * p.kcap + x.jlo) * D;
  const int nc = x.jhi - x.jlo;  // <= 32 PER
  float mine[PER];               // scores of candidates lane, lane + 32, ...
#pragma unroll
  for (int e = 0; e < PER; ++e) mine[e] = -INFINITY;
#pragma unroll
  for (int c0 = 0; c0 < 32 * PER; c0 += kBatch) {
    if (c0 >= nc) break;
    float v[kBatch][4];
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
#pragma unroll
      for (int t = 0; t < 4; ++t)
        v[u][t] = (c0 + u < nc && t < nt) ? kb[static_cast<long long>(c0 + u) * D + lane + 32 * t] : 0.f;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      float s = (qm[0] * v[u][0] + qm[1] * v[u][1]) + (qm[2] * v[u][2] + qm[3] * v[u][3]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(full, s, o);
      const int c = c0 + u;
      if (c < nc && lane == c % 32) mine[c / 32] = s;
    }
  }
  // rank among the candidates: larger first, ties to the lower index
  int rank[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) rank[e] = 0;
#pragma unroll
  for (int f = 0; f < PER; ++f) {
    if (32 * f >= nc) break;
    for (int m = 0; m < 32; ++m) {
      const float sm = __shfl_sync(full, mine[f], m);
      const int cm = 32 * f + m;
      if (cm >= nc) break;
#pragma unroll
      for (int e = 0; e < PER; ++e) {
        const int c = lane + 32 * e;
        rank[e] += (sm > mine[e] || (sm == mine[e] && cm < c)) ? 1 : 0;
      }
    }
  }
  const int k = k_count(p.permille, nc);
  int base = 0;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    const int c = lane + 32 * e;
    const bool sel = c < nc && rank[e] < k;
    const unsigned bal = __ballot_sync(full, sel);
    if (sel) list[base + __popc(bal & ((1u << lane) - 1u))] = x.jlo + c;
    base += __popc(bal);
  }
  for (int c = k + lane; c < p.kcap; c += 32) list[c] = -1;
  if (lane == 0) p.counts[x.row] = k;
}

// One CTA per (Q block i, query head h, sequence b), any number of K blocks.
__global__ void __launch_bounds__(kSelThreads) sparse_select_kernel(SparseParams p) {
  __shared__ float score[kSparseMaxKBlocks];
  __shared__ int flag[kSparseMaxKBlocks];
  __shared__ float qmean[128];
  __shared__ int warp_sum[kSelWarps];
  const int i = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const ListCtx x = list_ctx(p, b, h, i, t == 0);
  int32_t* list = p.blocks + x.row * p.kcap;
  if (x.empty) {
    for (int c = t; c < p.kcap; c += kSelThreads) list[c] = -1;
    if (t == 0) p.counts[x.row] = 0;
    return;
  }
  const int D = p.D, nk = x.nk;
  if (t < D) {
    const float* qs = q_halves(p, b, h, i);
    qmean[t] = (qs[t] + (x.has1 ? qs[D + t] : 0.f)) / x.nq;
  }
  __syncthreads();
  // Scores of the candidates: one warp per K block, lanes over the head dimension.
  const float* kb = p.kbar + (static_cast<long long>(b) * p.Hkv + h / p.G) * p.kcap * D;
  for (int j = x.jlo + warp; j < x.jhi; j += kSelWarps) {
    float s = 0.f;
    for (int d = lane; d < D; d += 32) s += qmean[d] * kb[static_cast<long long>(j) * D + d];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) score[j] = s;
  }
  __syncthreads();
  // Rank of every candidate's score (larger first, ties to the lower index);
  // the k best are selected.
  const int nc = x.jhi - x.jlo;
  const int k = k_count(p.permille, nc);
  for (int j = t; j < nk; j += kSelThreads) {
    int f = 0;
    if (j >= x.jlo && j < x.jhi) {
      const float sj = score[j];
      int rank = 0;
      for (int m = x.jlo; m < x.jhi; ++m) {
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
    for (int w = 0; w < kSelWarps; ++w) tot += warp_sum[w];
    base += tot;
    __syncthreads();
  }
  for (int c = k + t; c < p.kcap; c += kSelThreads) list[c] = -1;
  if (t == 0) p.counts[x.row] = k;
}

}  // namespace

cudaError_t launch_sparse_pool(const SparseParams& p, cudaStream_t s) {
  const dim3 grid(max(p.kcap, 2 * p.nqb), p.B, 2);
  if (p.H * p.D <= 1024)
    sparse_pool_kernel<512><<<grid, 512, 0, s>>>(p);
  else
    sparse_pool_kernel<256><<<grid, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_sparse_select(const SparseParams& p, cudaStream_t s) {
  const long long lists = static_cast<long long>(p.B) * p.H * p.nqb;
  const unsigned grid = static_cast<unsigned>((lists + kSelWarps - 1) / kSelWarps);
  if (p.kcap <= 32)
    sparse_select_warp_kernel<1><<<grid, kSelThreads, 0, s>>>(p);
  else if (p.kcap <= 64)
    sparse_select_warp_kernel<2><<<grid, kSelThreads, 0, s>>>(p);
  else if (p.kcap <= 128)
    sparse_select_warp_kernel<4><<<grid, kSelThreads, 0, s>>>(p);
  else
    sparse_select_kernel<<<dim3(p.nqb, p.H, p.B), kSelThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace jfa
