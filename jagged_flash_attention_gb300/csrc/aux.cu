// Device work-list scheduler, backward pre-pass (work lists, the row
// statistics LSE*log2e and Delta = rowsum(dO * O), zeroing of the broadcast
// fp32 dQ accumulator), dQ finalisation, and a fill kernel for the
// all-empty broadcast case.
#include "common.cuh"
#include "ptx.cuh"

namespace jfa {

namespace {

constexpr int kSchedThreads = 1024;
constexpr int kMaxBuckets = kSchedThreads;  // one bucket per thread in the scan

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

// Tiles of sequence b that become work items (one item per head and tile).
//  query items: tiles of `qrows` query rows (forward: 256 = two 128-row MMA
//            tiles; self-attention dQ pass: 128); self: of the sequence,
//            broadcast: of the dense Q
//  backward: key/value blocks of the sequence
__device__ __forceinline__ int n_tiles(const SchedParams& p, int L) {
  if (p.backward) return cdiv(L, kBN);
  // broadcast: every sequence, even an empty one, owns its output rows
  return p.broadcast ? cdiv(p.Lq, p.qrows) : cdiv(L, p.qrows);
}

// Cost bucket of sequence b: work of its longest item, in tile units.
//  forward:  key tiles a query tile visits (causal: the last query tile's)
//  backward: query tiles a key block visits (broadcast: all equal)
__device__ __forceinline__ int bucket_of(const SchedParams& p, int L) {
  int c = p.backward ? (p.broadcast ? 0 : cdiv(L, kBM)) : cdiv(L, kBN);
  return c < kMaxBuckets ? c : kMaxBuckets - 1;
}

// Block-wide exclusive scan over the buckets in DESCENDING bucket order:
// base[k] = sum of hist[k'] for k' > k.
__device__ void scan_desc(const int* hist, int* base, int* warp_tot) {
  const int tid = threadIdx.x;
  const int k = kMaxBuckets - 1 - tid;  // thread tid handles bucket k
  int v = hist[k];
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if ((tid & 31) >= o) x += y;
  }
  if ((tid & 31) == 31) warp_tot[tid >> 5] = x;
  __syncthreads();
  if (tid < 32) {
    int w = tid < static_cast<int>(blockDim.x >> 5) ? warp_tot[tid] : 0;
    int z = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, z, o);
      if (tid >= o) z += y;
    }
    warp_tot[tid] = z - w;  // exclusive warp prefix
  }
  __syncthreads();
  base[k] = warp_tot[tid >> 5] + x - v;
}

// Builds one work list with the whole block (kSchedThreads threads).
__device__ void sched_body(const SchedParams& p) {
  __shared__ int hist[kMaxBuckets];
  __shared__ int base[kMaxBuckets];
  __shared__ int cursor[kMaxBuckets];
  __shared__ int warp_tot[32];
  __shared__ int s_pos[kSchedThreads], s_nt[kSchedThreads];
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  for (int i = tid; i < kMaxBuckets; i += blockDim.x) hist[i] = 0, cursor[i] = 0;
  if (tid == 0) s_bad = (p.offsets[0] != 0);
  __syncthreads();
  for (int b = tid; b < p.B; b += blockDim.x) {
    const int L = p.offsets[b + 1] - p.offsets[b];
    if (L < 0 || L > p.max_len) {
      s_bad = 1;
      continue;
    }
    const int nt = n_tiles(p, L);
    if (nt > 0) atomicAdd(&hist[bucket_of(p, L)], p.H * nt);
  }
  __syncthreads();
  if (s_bad) {
    if (tid == 0) {
      p.hdr->n_items = 0;
      p.hdr->T = 0;
      p.hdr->ticket = 0;
      p.hdr->valid = 0;
      atomicOr(p.err, kErrBadOffsets);
    }
    return;
  }
  scan_desc(hist, base, warp_tot);
  __syncthreads();
  const int total = base[0] + hist[0];
  if (total > p.capacity) {
    if (tid == 0) {
      p.hdr->n_items = 0;
      p.hdr->T = 0;
      p.hdr->ticket = 0;
      p.hdr->valid = 0;
      atomicOr(p.err, kErrCapacity);
    }
    return;
  }
  // Chunks of blockDim sequences.  Each thread reserves the slots of one
  // sequence; threads of a warp whose sequences fall in the same cost bucket
  // do it with one shared atomic (many short sequences share a few buckets).
  // Then each warp writes the items of its share of the chunk's sequences,
  // lanes over items.  Heads outer, tiles inner, so that consecutive items
  // share K/V (or Q) in L2; forward causal: longest query tile first.
  const int lane = tid & 31, nwarps = blockDim.x >> 5;
  const bool reverse = !p.backward && p.causal;
  for (int c0 = 0; c0 < p.B; c0 += blockDim.x) {
    const int b = c0 + tid;
    int nt = 0, n = 0, key = 0;
    if (b < p.B) {
      const int L = p.offsets[b + 1] - p.offsets[b];
      nt = n_tiles(p, L);
      n = p.H * nt;
      key = bucket_of(p, L);
    }
    const unsigned active = __ballot_sync(0xffffffffu, n > 0);
    int pos = 0;
    if (n > 0) {
      const unsigned peers = __match_any_sync(active, key);
      const int leader = __ffs(peers) - 1;
      int pre = 0, tot = 0;
      for (unsigned m = peers; m; m &= m - 1) {
        const int j = __ffs(m) - 1;
        const int nj = __shfl_sync(peers, n, j);
        tot += nj;
        if (j < lane) pre += nj;
      }
      int first = 0;
      if (lane == leader) first = atomicAdd(&cursor[key], tot);
      first = __shfl_sync(peers, first, leader);
      pos = base[key] + first + pre;
    }
    s_pos[tid] = pos;
    s_nt[tid] = nt;
    __syncthreads();
    for (int w = tid >> 5; w < kSchedThreads && c0 + w < p.B; w += nwarps) {
      const int ntl = s_nt[w];
      if (ntl == 0) continue;
      const int nl = p.H * ntl, pl = s_pos[w];
      for (int j = lane; j < nl; j += 32) {
        const int h = j / ntl, t = j - h * ntl;
        const int tt = reverse ? ntl - 1 - t : t;
        p.items[pl + j] = make_int2(c0 + w, (h << 16) | tt);
      }
    }
    __syncthreads();
  }
  if (tid == 0) {
    p.hdr->n_items = total;
    p.hdr->T = p.offsets[p.B];
    p.hdr->ticket = 0;
    p.hdr->valid = 1;
  }
}

__global__ void __launch_bounds__(kSchedThreads) sched_kernel(SchedParams p) { sched_body(p); }

constexpr float kLog2e = 1.4426950408889634f;

// Row statistics of the backward pass with blocks [0, nblk) of the caller's
// grid: Delta[row] = sum_d dO[row, d] * O[row, d] in fp32 (the rowsum the
// gradient of the softmax subtracts), and for self-attention LSE*log2e next
// to it.  tpr = D/8 threads per row, each reading 16 bytes of both tensors;
// kUnroll rows per thread in flight.
constexpr int kUnroll = 2;      // broadcast-Q rows in flight per thread
constexpr int kUnrollSelf = 1;  // self-attention steps in flight per warp (32-byte loads)

__device__ void stats_body(const PrepParams& p, long long blk, long long nblk) {
  long long rows;
  int T = 0;
  if (p.broadcast) {
    rows = static_cast<long long>(p.B) * p.Lq * p.H;
  } else {
    // T is validated by the scheduler blocks; here it only has to keep the
    // reads inside the caller's Tcap rows.
    T = p.offsets[p.B];
    if (T < 0 || T > p.Tcap) return;
    rows = static_cast<long long>(T) * p.H;
  }
  if (!p.broadcast && blk == 0) {
    // Positions of rows before 0, read by boxes that start early: zeros (a
    // finite Delta for the columns those boxes mask).
    for (int i = threadIdx.x; i < kStatCopies * kStatPad; i += blockDim.x) {
      const int k = i / kStatPad;
      const long long u = i % kStatPad;
      if (u < stat_pos(0, k)) {
        float* f = p.stat + k * p.stat_stride + stat_float(u);
        f[0] = 0.f;
        f[4] = 0.f;
      }
    }
  }
  const int tpr = p.D / 8;
  const int rpw = 32 / tpr;  // rows per warp and unroll step
  const int lane = threadIdx.x & 31;
  const int part = lane % tpr;
  const long long wid = (blk * blockDim.x + threadIdx.x) >> 5;
  if (!p.broadcast) {
    // Self-attention: a warp takes 32 consecutive rows r0.. of O and dO in
    // memory order (row = t*H + h), one contiguous block (D/16 threads per
    // row, 32 bytes of O and dO each, 32/(D/16) rows per step); the row sums
    // are gathered so that lane l ends with row r0 + l, and the statistics
    // of lanes with the same head land on consecutive tokens.
    const int tpr32 = p.D / 16, rpw32 = 32 / tpr32, part32 = lane % tpr32;
    const bool v8 = ((reinterpret_cast<uintptr_t>(p.out) | reinterpret_cast<uintptr_t>(p.dout)) & 31) == 0;
    const long long nwarps = (nblk * blockDim.x) >> 5;
    for (long long r0 = wid * 32; r0 < rows; r0 += nwarps * 32) {
      float mine = 0.f;
      for (int s0 = 0; s0 < 32; s0 += rpw32 * kUnrollSelf) {
        uint32_t o[kUnrollSelf][8], g[kUnrollSelf][8];
#pragma unroll
        for (int u = 0; u < kUnrollSelf; ++u) {
          const long long row = r0 + s0 + u * rpw32 + lane / tpr32;
          if (row < rows) {
            const __nv_bfloat16* po = p.out + row * p.D + part32 * 16;
            const __nv_bfloat16* pg = p.dout + row * p.D + part32 * 16;
            if (v8) {
              ld_global_v8(po, o[u]);
              ld_global_v8(pg, g[u]);
            } else {  // the caller's buffers are only 16-byte aligned
              const uint4 o0 = reinterpret_cast<const uint4*>(po)[0], o1 = reinterpret_cast<const uint4*>(po)[1];
              const uint4 g0 = reinterpret_cast<const uint4*>(pg)[0], g1 = reinterpret_cast<const uint4*>(pg)[1];
              o[u][0] = o0.x, o[u][1] = o0.y, o[u][2] = o0.z, o[u][3] = o0.w;
              o[u][4] = o1.x, o[u][5] = o1.y, o[u][6] = o1.z, o[u][7] = o1.w;
              g[u][0] = g0.x, g[u][1] = g0.y, g[u][2] = g0.z, g[u][3] = g0.w;
              g[u][4] = g1.x, g[u][5] = g1.y, g[u][6] = g1.z, g[u][7] = g1.w;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) o[u][i] = g[u][i] = 0u;
          }
        }
#pragma unroll
        for (int u = 0; u < kUnrollSelf; ++u) {
          float acc = 0.f;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&o[u][i]));
            const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&g[u][i]));
            acc = fmaf(a.x, c.x, acc);
            acc = fmaf(a.y, c.y, acc);
          }
          for (int off = tpr32 / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
          // row s0 + u*rpw32 + j sits in lanes [j*tpr32, (j+1)*tpr32); lane l keeps row l
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (j >= rpw32) break;
            const float v = __shfl_sync(0xffffffffu, acc, j * tpr32);
            if (lane == s0 + u * rpw32 + j) mine = v;
          }
        }
      }
      const long long row = r0 + lane;
      if (row < rows) {
        const long long t = row / p.H, h = row % p.H;
        const long long si = h * T + t;
        const float nl = -p.lse[si] * kLog2e;
#pragma unroll
        for (int k = 0; k < kStatCopies; ++k) {
          float* f = p.stat + k * p.stat_stride + stat_float(stat_pos(si, k));
          f[0] = nl;
          f[4] = -mine;
        }
      }
    }
    return;
  }
  const long long nw = (nblk * blockDim.x) >> 5;
  const long long step = static_cast<long long>(rpw) * kUnroll;
  for (long long r0 = wid * step; r0 < rows; r0 += nw * step) {
    uint4 o[kUnroll], g[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const long long row = r0 + u * rpw + lane / tpr;
      if (row < rows) {
        o[u] = *reinterpret_cast<const uint4*>(p.out + row * p.D + part * 8);
        g[u] = *reinterpret_cast<const uint4*>(p.dout + row * p.D + part * 8);
      } else {
        o[u] = make_uint4(0, 0, 0, 0);
        g[u] = o[u];
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&o[u]);
      const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g[u]);
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 a = __bfloat1622float2(o2[i]);
        const float2 c = __bfloat1622float2(g2[i]);
        acc = fmaf(a.x, c.x, acc);
        acc = fmaf(a.y, c.y, acc);
      }
      for (int off = tpr / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      const long long row = r0 + u * rpw + lane / tpr;
      if (row < rows && part == 0) {
        if (p.broadcast) {
          const long long h = row % p.H;
          const long long bi = row / p.H;  // b * Lq + i
          const long long b = bi / p.Lq, i = bi % p.Lq;
          p.delta[(b * p.H + h) * p.Lq + i] = acc;
        } else {
          const long long h = row % p.H, t = row / p.H;
          const long long si = h * T + t;
          const float nl = -p.lse[si] * kLog2e;
#pragma unroll
          for (int k = 0; k < kStatCopies; ++k) {
            float* f = p.stat + k * p.stat_stride + stat_float(stat_pos(si, k));
            f[0] = nl;
            f[4] = -acc;
          }
        }
      }
    }
  }
}

// Backward pre-pass: work lists (blocks [0, n_sched)), row statistics and,
// for broadcast-Q, zeroing of the fp32 dQ accumulator (the other blocks).
__global__ void __launch_bounds__(kSchedThreads) bwd_prep_kernel(const __grid_constant__ PrepParams p) {
  if (blockIdx.x < p.n_sched) {
    if (blockIdx.x == 0)
      sched_body(p.sched[0]);
    else
      sched_body(p.sched[1]);
    return;
  }
  const long long blk = blockIdx.x - p.n_sched, nblk = gridDim.x - p.n_sched;
  stats_body(p, blk, nblk);
  if (p.broadcast) {
    const long long gtid = blk * blockDim.x + threadIdx.x;
    float4* z = reinterpret_cast<float4*>(p.dq_acc);
    for (long long i = gtid; i < p.dq_acc_elems_bcast / 4; i += nblk * blockDim.x)
      z[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// dq = bf16(scale * sum over shards of the fp32 accumulator)
__global__ void __launch_bounds__(256) finalize_kernel(FinParams p) {
  const long long n = p.broadcast ? (long long)p.Lq * p.H * p.D
                                  : (p.hdr->valid ? (long long)p.hdr->T * p.H * p.D : 0);
  const long long gtid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  for (long long i = gtid; i < n / 4; i += nthreads) {
    float4 a = reinterpret_cast<const float4*>(p.dq_acc)[i];
    for (int s = 1; s < p.shards; ++s) {
      const float4 c = reinterpret_cast<const float4*>(p.dq_acc + s * p.shard_stride)[i];
      a.x += c.x, a.y += c.y, a.z += c.z, a.w += c.w;
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(a.x * p.scale, a.y * p.scale);
    __nv_bfloat162 hi = __floats2bfloat162_rn(a.z * p.scale, a.w * p.scale);
    uint2 v;
    v.x = *reinterpret_cast<uint32_t*>(&lo);
    v.y = *reinterpret_cast<uint32_t*>(&hi);
    reinterpret_cast<uint2*>(p.dq)[i] = v;
  }
}

// out[rows, D] = 0 (bf16), lse[rows] = -inf: outputs of a broadcast batch
// whose sequences are all empty.
__global__ void fill_empty_kernel(__nv_bfloat16* out, float* lse, long long rows, int D) {
  const long long gtid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long nthreads = (long long)gridDim.x * blockDim.x;
  for (long long i = gtid; i < rows * D / 8; i += nthreads)
    reinterpret_cast<uint4*>(out)[i] = make_uint4(0, 0, 0, 0);
  if (lse)
    for (long long i = gtid; i < rows; i += nthreads) lse[i] = -INFINITY;
}

}  // namespace

cudaError_t launch_sched(const SchedParams& p, cudaStream_t s) {
  sched_kernel<<<1, kSchedThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_prep(const PrepParams& p, int sms, cudaStream_t s) {
  bwd_prep_kernel<<<p.n_sched + sms * 2, kSchedThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const FinParams& p, int sms, cudaStream_t s) {
  finalize_kernel<<<sms * 8, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fill_empty(__nv_bfloat16* out, float* lse, long long rows, int D,
                              cudaStream_t s) {
  fill_empty_kernel<<<256, 256, 0, s>>>(out, lse, rows, D);
  return cudaGetLastError();
}

}  // namespace jfa
