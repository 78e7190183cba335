// Device work-list schedulers, backward pre-pass (work lists and the row
// statistics LSE*log2e and Delta = rowsum(dO * O)), the broadcast dQ
// finalisation, and a fill kernel for the all-empty broadcast case.
#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"

namespace jfa {

namespace {

constexpr int kSchedThreads = 1024;
constexpr int kQbSmemOff = 8192;  // key-tile prefix entries kept in shared memory
constexpr int kMaxBuckets = kSchedThreads;  // one bucket per thread in the scan

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

// Tiles of sequence b that become work items (one item per head and tile).
//  query items: tiles of `qrows` query rows (forward: 256 = two 128-row MMA
//            tiles; self-attention dQ pass: 128); self: of the sequence,
//            broadcast: of the dense Q
//  backward: key/value blocks of the sequence (pairs of them for CTA pairs)
__device__ __forceinline__ int n_tiles(const SchedParams& p, int L) {
  if (p.backward) return cdiv(L, kBN * p.kpair);
  // broadcast: every sequence, even an empty one, owns its output rows
  return p.broadcast ? cdiv(p.Lq, p.qrows) : cdiv(L, p.qrows);
}

// Cost bucket of sequence b: work of its longest item, in tile units.
//  forward:  key tiles a query tile visits (causal: the last query tile's)
//  backward: query tiles a key block visits (broadcast: all equal)
// A sliding window bounds both by the band's width.
__device__ __forceinline__ int bucket_of(const SchedParams& p, int L) {
  int c = p.backward ? (p.broadcast ? 0 : cdiv(L, kBM)) : cdiv(L, kBN);
  if (p.causal) {
    const long long w = static_cast<long long>(p.wl) + p.wr + (p.backward ? kBN : p.qrows);
    if (w < L) c = min(c, static_cast<int>(w / kBN) + 2);
  }
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
// Thread tid handles sequences tid, tid + blockDim, ...; the lengths of the
// first kPer of them stay in registers between the two passes, loaded
// together so that their latencies overlap.
constexpr int kPer = 8;
struct SchedSmem {
  int hist[kMaxBuckets], base[kMaxBuckets], cursor[kMaxBuckets];
  int warp_tot[32];
  int bad, badblk, nbig;
  int4 big[kSchedThreads];  // sequences with many items: {b, pos, tiles, items}
};
__device__ void sched_body(const SchedParams& p, SchedSmem& sm) {
  int* hist = sm.hist;
  int* base = sm.base;
  int* cursor = sm.cursor;
  int* warp_tot = sm.warp_tot;
  int& s_bad = sm.bad;
  int& s_nbig = sm.nbig;
  int4* s_big = sm.big;
  const int tid = threadIdx.x, lane = tid & 31;
  for (int i = tid; i < kMaxBuckets; i += blockDim.x) hist[i] = 0, cursor[i] = 0;
  if (tid == 0) {
    s_bad = (p.offsets[0] != 0);
    sm.badblk = 0;
  }
  int Lr[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int b = i * blockDim.x + tid;
    Lr[i] = b < p.B ? p.offsets[b + 1] - p.offsets[b] : 0;
  }
  auto length = [&](int i, int b) {  // sequence b = i * blockDim + tid
    int L = 0;
#pragma unroll
    for (int k = 0; k < kPer; ++k)
      if (k == i) L = Lr[k];
    return i < kPer ? L : p.offsets[b + 1] - p.offsets[b];
  };
  __syncthreads();
  // Lanes of a warp whose sequences share a cost bucket add to it with one
  // shared atomic (thousands of short sequences fall into a few buckets, and
  // same-address atomics serialise).
  for (int i = 0; i * static_cast<int>(blockDim.x) < p.B; ++i) {
    const int b = i * blockDim.x + tid;
    int n = 0, key = -1;
    if (b < p.B) {
      const int L = length(i, b);
      if (L < 0 || L > p.max_len) {
        s_bad = 1;
      } else {
        n = p.H * n_tiles(p, L);
        if (n > 0) key = bucket_of(p, L);
      }
    }
    const unsigned active = __ballot_sync(0xffffffffu, key >= 0);
    if (key >= 0) {
      const unsigned peers = __match_any_sync(active, key);
      int tot = 0;
      for (unsigned m = peers; m; m &= m - 1) tot += __shfl_sync(peers, n, __ffs(m) - 1);
      if (lane == __ffs(peers) - 1) atomicAdd(&hist[key], tot);
    }
  }
  // Block lists of the sparse forward: the results list_check_kernel wrote
  // just before (anything but 1, even a slot never written, is a bad list).
  if (p.blocks != nullptr) {
    for (int v = tid; v < p.n_check; v += blockDim.x)
      if (p.check[v] != 1) sm.badblk = 1;
  }
  __syncthreads();
  if (s_bad || sm.badblk) {
    if (tid == 0) {
      p.hdr->n_items = 0;
      p.hdr->T = 0;
      p.hdr->ticket = 0;
      p.hdr->valid = 0;
      atomicOr(p.err, s_bad ? kErrBadOffsets : kErrBadBlocks);
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
  // Each thread reserves the slots of its sequence; threads of a warp whose
  // sequences fall in the same cost bucket do it with one shared atomic.  A
  // thread writes the items of its own sequence if they are few; sequences
  // with many items go to a shared list that all warps then write, lanes
  // over items.  Heads outer, tiles inner, so that consecutive items share
  // K/V (or Q) in L2; forward causal: longest query tile first.
  const bool reverse = !p.backward && p.causal;
  // Broadcast dK/dV list: heads outermost over the whole list (every item
  // costs the same), so that a CTA's consecutive items share the head and
  // with it the dense Q tiles its shared memory still holds.  Every
  // sequence's block of items is H * tiles long, so pos / H is the offset of
  // its tiles within one head's part.
  const bool head_outer = p.broadcast && p.backward;
  const int per_head = total / p.H;
  auto slot = [&](int pos, int h, int t, int nt) {
    return head_outer ? h * per_head + pos / p.H + t : pos + h * nt + t;
  };
  constexpr int kOwnItems = 32;  // at most this many: written by the thread itself
  for (int i = 0; i * static_cast<int>(blockDim.x) < p.B; ++i) {
    if (tid == 0) s_nbig = 0;
    __syncthreads();
    const int b = i * blockDim.x + tid;
    int nt = 0, n = 0, key = 0;
    if (b < p.B) {
      const int L = length(i, b);
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
    if (n > 0 && n <= kOwnItems) {
      for (int h = 0; h < p.H; ++h)
        for (int t = 0; t < nt; ++t)
          p.items[slot(pos, h, t, nt)] = make_int2(b, (h << 16) | (reverse ? nt - 1 - t : t));
    } else if (n > kOwnItems) {
      s_big[atomicAdd(&s_nbig, 1)] = make_int4(b, pos, nt, n);
    }
    __syncthreads();
    for (int k = tid >> 5; k < s_nbig; k += blockDim.x >> 5) {
      const int4 g = s_big[k];
      for (int j = lane; j < g.w; j += 32) {
        const int h = j / g.z, t = j - h * g.z;
        p.items[slot(g.y, h, t, g.z)] = make_int2(g.x, (h << 16) | (reverse ? g.z - 1 - t : t));
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

// List r of the sparse forward (sequence b, head, 256-row query block i): a
// count of at most the sequence's key tiles and strictly ascending key tiles
// below it.  Lists of query blocks past the sequence (broadcast: of every
// sequence, the dense Q's blocks) are not read, nor those of sequences with
// bad offsets (which the scheduler itself rejects).
__device__ bool list_ok(const SchedParams& p, long long r) {
  const int i = static_cast<int>(r % p.nqb);
  const int b = static_cast<int>(r / p.nqb / p.H);
  const int L = p.offsets[b + 1] - p.offsets[b];
  if (L < 0 || L > p.max_len || i * kFwdRows >= (p.broadcast ? p.Lq : L)) return true;
  const int nk = cdiv(L, kBN);
  const int c = p.counts[r];
  bool ok = c >= 0 && c <= nk;
  const int32_t* lst = p.blocks + r * p.kcap;
  const int n = ok ? c : 0;
  // entries in groups of 8 loaded together (no exit between them, so the
  // loads of a group are in flight at once)
  int prev = -1;
  for (int e0 = 0; e0 < n; e0 += 8) {
    int v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = e0 + q < n ? lst[e0 + q] : nk + 1;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (e0 + q < n) {
        ok = ok && v[q] > prev && v[q] < nk;
        prev = v[q];
      }
    }
  }
  return ok;
}

// Checks every list of the sparse forward, a thread per list; block x
// writes check[x] = 1 when all its lists are valid, 2 otherwise.
constexpr int kCheckThreads = 256;
__global__ void __launch_bounds__(kCheckThreads) list_check_kernel(SchedParams p) {
  const long long n_lists = static_cast<long long>(p.B) * p.H * p.nqb;
  bool bad = false;
  for (long long r = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; r < n_lists;
       r += static_cast<long long>(gridDim.x) * blockDim.x)
    bad = bad || !list_ok(p, r);
  bad = __syncthreads_or(bad ? 1 : 0) != 0;
  if (threadIdx.x == 0) p.check[blockIdx.x] = bad ? 2 : 1;
}

struct QbSmem {
  int warp_tot[32];
  int bad, carry;
  int kt[kQbSmemOff];  // key-tile prefix, when B + 1 <= kQbSmemOff
};
// The two list builders never run in the same block: one static buffer.
union SchedScratch {
  SchedSmem s;
  QbSmem q;
};

__global__ void __launch_bounds__(kSchedThreads) sched_kernel(SchedParams p) {
  __shared__ SchedScratch sm;
  sched_body(p, sm.s);
}

// A built work list copied out as 4 ints per item, with its item count
// (and, for the broadcast dQ-pass list, its chunk count): list inspection
// for tests.  Forward and backward lists: {b, h, tile, 0}; broadcast dQ
// pass: {h | pair << 16, b, j, n}.  count[0] = -1 if the list is invalid.
__global__ void export_list_kernel(const WorkHeader* hdr, const void* items, int qb, int32_t* out,
                                   int capacity, int32_t* count) {
  const int n = hdr->valid ? hdr->n_items : 0;
  const int gtid = blockIdx.x * blockDim.x + threadIdx.x;
  if (gtid == 0) {
    count[0] = hdr->valid ? n : -1;
    count[1] = qb ? hdr->n_chunks : 0;
  }
  for (int i = gtid; i < n && i < capacity; i += gridDim.x * blockDim.x) {
    int4 v;
    if (qb) {
      const QbItem it = static_cast<const QbItem*>(items)[i];
      v = make_int4(it.hp, it.b, it.j, it.n);
    } else {
      const Item it = static_cast<const Item*>(items)[i];
      v = make_int4(it.x, it.y >> 16, it.y & 0xffff, 0);
    }
    reinterpret_cast<int4*>(out)[i] = v;
  }
}

// Inclusive prefix sum over the block (blockDim a multiple of 32, at most
// 1024); warp_tot: 32 ints of shared memory.
__device__ int block_incl_scan(int v, int* warp_tot) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_tot[w] = x;
  __syncthreads();
  if (w == 0) {
    int t = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += y;
    }
    warp_tot[lane] = t;
  }
  __syncthreads();
  const int r = x + (w > 0 ? warp_tot[w - 1] : 0);
  __syncthreads();
  return r;
}

// Work list of the broadcast-Q dQ pass with the whole block: the key tiles
// of all sequences, in order, form one stream per (head, query-tile pair);
// it is cut into nc equal chunks, and item (c, h, pair) at list index
// (c * H + h) * pairs + pair starts at the sequence and tile where chunk c
// starts.  kt_off[b] = key tiles of the sequences before b.
__device__ void qb_sched_body(const QbSchedParams& p, QbSmem& sm) {
  int* warp_tot = sm.warp_tot;
  int& s_bad = sm.bad;
  int& s_carry = sm.carry;
  const int tid = threadIdx.x;
  if (tid == 0) {
    s_bad = (p.offsets[0] != 0);
    s_carry = 0;
  }
  __syncthreads();
  for (int b0 = 0; b0 < p.B; b0 += blockDim.x) {
    const int b = b0 + tid;
    int nt = 0;
    if (b < p.B) {
      const int L = p.offsets[b + 1] - p.offsets[b];
      if (L < 0 || L > p.max_len)
        s_bad = 1;
      else
        nt = cdiv(L, kBN);
    }
    const int incl = block_incl_scan(nt, warp_tot);
    if (b < p.B) p.kt_off[b] = s_carry + incl - nt;
    __syncthreads();
    if (tid == blockDim.x - 1) s_carry += incl;
    __syncthreads();
  }
  const int total = s_carry;
  if (tid == 0) p.kt_off[p.B] = total;
  __syncthreads();  // kt_off visible to the whole block
  const int pairs = cdiv(p.Lq, kQbRows);
  const int nc = s_bad ? 0 : min(p.chunk_cap, (total + 3) / 4);
  const long long n_items = static_cast<long long>(nc) * p.H * pairs;
  if (s_bad || n_items > p.capacity) {
    if (tid == 0) {
      p.hdr->n_items = 0;
      p.hdr->n_chunks = 0;
      p.hdr->T = 0;
      p.hdr->ticket = 0;
      p.hdr->valid = 0;
      atomicOr(p.err, s_bad ? kErrBadOffsets : kErrCapacity);
    }
    return;
  }
  // Chunk starts: the last sequence b with kt_off[b] <= s0 (it is
  // non-empty), by binary search over kt_off; a copy in shared memory when
  // it fits.
  int* s_kt = sm.kt;
  const bool in_smem = p.B + 1 <= kQbSmemOff;
  if (in_smem)
    for (int b = tid; b <= p.B; b += blockDim.x) s_kt[b] = p.kt_off[b];
  __syncthreads();
  const int* kt = in_smem ? s_kt : p.kt_off;
  for (int idx = tid; idx < n_items; idx += blockDim.x) {
    const int c = idx / (p.H * pairs);
    const int rem = idx - c * (p.H * pairs);
    const int h = rem / pairs, pair = rem - h * pairs;
    const int s0 = static_cast<int>(static_cast<long long>(c) * total / nc);
    const int s1 = static_cast<int>(static_cast<long long>(c + 1) * total / nc);
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (kt[mid] <= s0)
        lo = mid;
      else
        hi = mid - 1;
    }
    QbItem it;
    it.hp = h | (pair << 16);
    it.b = lo;
    it.j = s0 - kt[lo];
    it.n = s1 - s0;
    p.items[idx] = it;
  }
  if (tid == 0) {
    p.hdr->n_items = static_cast<int>(n_items);
    p.hdr->n_chunks = nc;
    p.hdr->T = p.offsets[p.B];
    p.hdr->ticket = 0;
    p.hdr->valid = 1;
  }
}

constexpr float kLog2e = 1.4426950408889634f;

// Row statistics of the backward pass with blocks [0, nblk) of the caller's
// grid: Delta[row] = sum_d dO[row, d] * O[row, d] in fp32 (the rowsum the
// gradient of the softmax subtracts) and LSE*log2e, stored as {-LSE*log2e,
// -Delta}.  Self-attention rows (t, h) go to every copy at position h*T + t;
// broadcast rows (b, i, h) to position (b*H + h)*lq_pad + i.  A warp takes 32
// consecutive rows r0.. of O and dO in memory order (one contiguous block;
// D/16 threads per row, 32 bytes of O and dO each, 32/(D/16) rows per step);
// the row sums are gathered so that lane l ends with row r0 + l.
__device__ void stats_body(const PrepParams& p, long long blk, long long nblk) {
  long long rows;
  int T = 0;
  const long long lq_pad = static_cast<long long>(cdiv(p.Lq, kBM)) * kBM;
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
  const int lane = threadIdx.x & 31;
  const long long wid = (blk * blockDim.x + threadIdx.x) >> 5;
  const int tpr32 = p.D / 16, rpw32 = 32 / tpr32;
  const bool v8 = ((reinterpret_cast<uintptr_t>(p.out) | reinterpret_cast<uintptr_t>(p.dout)) & 31) == 0;
  const long long nwarps = (nblk * blockDim.x) >> 5;
  for (long long r0 = wid * 32; r0 < rows; r0 += nwarps * 32) {
    // This lane's row: its LSE is loaded first, independently of O and dO.
    const long long row = r0 + lane;
    long long pos = 0;  // statistics position (self: before the copy offset)
    float nl = 0.f;
    if (row < rows) {
      const long long h = row % p.H, t = row / p.H;
      if (p.broadcast) {
        const long long b = t / p.Lq, i = t - b * p.Lq;
        pos = (b * p.H + h) * lq_pad + i;
        nl = -p.lse[(b * p.H + h) * p.Lq + i] * kLog2e;
      } else {
        pos = h * T + t;
        nl = -p.lse[pos] * kLog2e;
      }
    }
    float mine = 0.f;
    for (int s0 = 0; s0 < 32; s0 += rpw32) {
      uint32_t o[8], g[8];
      const long long rr = r0 + s0 + lane / tpr32;
      const int part32 = lane % tpr32;
      if (rr < rows) {
        const __nv_bfloat16* po = p.out + rr * p.D + part32 * 16;
        const __nv_bfloat16* pg = p.dout + rr * p.D + part32 * 16;
        if (v8) {
          ld_global_v8(po, o);
          ld_global_v8(pg, g);
        } else {  // the caller's buffers are only 16-byte aligned
          const uint4 o0 = reinterpret_cast<const uint4*>(po)[0], o1 = reinterpret_cast<const uint4*>(po)[1];
          const uint4 g0 = reinterpret_cast<const uint4*>(pg)[0], g1 = reinterpret_cast<const uint4*>(pg)[1];
          o[0] = o0.x, o[1] = o0.y, o[2] = o0.z, o[3] = o0.w;
          o[4] = o1.x, o[5] = o1.y, o[6] = o1.z, o[7] = o1.w;
          g[0] = g0.x, g[1] = g0.y, g[2] = g0.z, g[3] = g0.w;
          g[4] = g1.x, g[5] = g1.y, g[6] = g1.z, g[7] = g1.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = g[i] = 0u;
      }
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&o[i]));
        const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&g[i]));
        acc = fmaf(a.x, c.x, acc);
        acc = fmaf(a.y, c.y, acc);
      }
      for (int off = tpr32 / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      // row s0 + j sits in lanes [j*tpr32, (j+1)*tpr32); lane l keeps row l
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j >= rpw32) break;
        const float v = __shfl_sync(0xffffffffu, acc, j * tpr32);
        if (lane == s0 + j) mine = v;
      }
    }
    if (row < rows) {
      if (p.broadcast) {
        float* f = p.stat + stat_float(pos);
        f[0] = nl;
        f[4] = -mine;
      } else {
#pragma unroll
        for (int k = 0; k < kStatCopies; ++k) {
          float* f = p.stat + k * p.stat_stride + stat_float(stat_pos(pos, k));
          f[0] = nl;
          f[4] = -mine;
        }
      }
    }
  }
}

// Backward pre-pass: work lists (blocks [0, n_sched)), then the row
// statistics (the other blocks).  Broadcast-Q: block 1 builds the dQ-pass
// list, and the padding rows of the statistics (rows q_len.. of each
// sequence's last query tile) get {-inf, 0}, so that P = 0 there.
__global__ void __launch_bounds__(kSchedThreads) bwd_prep_kernel(const __grid_constant__ PrepParams p) {
  if (blockIdx.x < p.n_sched) {
    __shared__ SchedScratch sm;
    if (blockIdx.x == 0 && p.qb_only)
      qb_sched_body(p.qb, sm.q);
    else if (blockIdx.x == 0)
      sched_body(p.sched[0], sm.s);
    else if (p.broadcast)
      qb_sched_body(p.qb, sm.q);
    else
      sched_body(p.sched[1], sm.s);
    return;
  }
  const long long blk = blockIdx.x - p.n_sched, nblk = gridDim.x - p.n_sched;
  stats_body(p, blk, nblk);
  if (p.broadcast) {
    const int lq_pad = cdiv(p.Lq, kBM) * kBM, npad = lq_pad - p.Lq;
    const long long n = static_cast<long long>(p.B) * p.H * npad;
    for (long long i = blk * blockDim.x + threadIdx.x; i < n; i += nblk * blockDim.x) {
      const long long bh = i / npad, k = i - bh * npad;
      float* f = p.stat + stat_float(bh * lq_pad + p.Lq + k);
      f[0] = -INFINITY;
      f[4] = 0.f;
    }
  }
}

__global__ void __launch_bounds__(kSchedThreads) qb_sched_kernel(QbSchedParams p) {
  __shared__ SchedScratch sm;
  qb_sched_body(p, sm.q);
}

// Broadcast dQ: dq[l, h, :] = bf16(scale * sum over the chunks c of the
// partial of item (c, h, pair = l / 256)).  A block takes 32 four-column
// groups (l, h, d4) and splits the chunks among kFinGroups thread groups;
// group g sums chunks g, g + kFinGroups, ..., and the group sums are added in
// group order, so the result does not depend on timing.
constexpr int kFinGroups = 8;
constexpr int kFinThreads = 32 * kFinGroups;
__global__ void __launch_bounds__(kFinThreads) finalize_kernel(FinParams p) {
  __shared__ float4 part_sum[kFinGroups][32];
  if (!p.hdr->valid) return;
  const int nc = p.hdr->n_chunks;
  const int pairs = cdiv(p.Lq, kQbRows);
  const int d4n = p.D / 4;
  const long long n = static_cast<long long>(p.Lq) * p.H * d4n;
  const int e = threadIdx.x & 31, grp = threadIdx.x >> 5;
  for (long long i0 = static_cast<long long>(blockIdx.x) * 32; i0 < n;
       i0 += static_cast<long long>(gridDim.x) * 32) {
    const long long i = i0 + e;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i < n) {
      const int d4 = static_cast<int>(i % d4n);
      const long long lh = i / d4n;
      const int h = static_cast<int>(lh % p.H), l = static_cast<int>(lh / p.H);
      const int pair = l / kQbRows, g = (l % kQbRows) / kBM, r = l % kBM;
      const long long stride = static_cast<long long>(kFinGroups) * p.H * pairs * 2 * kBM * p.D;
      const float* src = p.part + ((((static_cast<long long>(grp) * p.H + h) * pairs + pair) * 2 + g) * kBM + r) * p.D + 4 * d4;
#pragma unroll 4
      for (int c = grp; c < nc; c += kFinGroups, src += stride) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        a.x += v.x, a.y += v.y, a.z += v.z, a.w += v.w;
      }
    }
    part_sum[grp][e] = a;
    __syncthreads();
    if (grp == 0 && i < n) {
      for (int q = 1; q < kFinGroups; ++q) {
        const float4 v = part_sum[q][e];
        a.x += v.x, a.y += v.y, a.z += v.z, a.w += v.w;
      }
      __nv_bfloat162 lo = __floats2bfloat162_rn(a.x * p.scale, a.y * p.scale);
      __nv_bfloat162 hi = __floats2bfloat162_rn(a.z * p.scale, a.w * p.scale);
      uint2 v;
      v.x = *reinterpret_cast<uint32_t*>(&lo);
      v.y = *reinterpret_cast<uint32_t*>(&hi);
      reinterpret_cast<uint2*>(p.dq)[i] = v;
    }
    __syncthreads();
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

int list_check_blocks(const SchedParams& p) {
  const long long lists = static_cast<long long>(p.B) * p.H * p.nqb;
  return static_cast<int>(std::max(1LL, std::min(1024LL, (lists + kCheckThreads - 1) / kCheckThreads)));
}

cudaError_t launch_list_check(const SchedParams& p, cudaStream_t s) {
  list_check_kernel<<<p.n_check, kCheckThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_sched(const SchedParams& p, cudaStream_t s) {
  sched_kernel<<<1, kSchedThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_qb_sched(const QbSchedParams& p, cudaStream_t s) {
  qb_sched_kernel<<<1, kSchedThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_export_list(const WorkHeader* hdr, const void* items, int qb, int32_t* out,
                               int capacity, int32_t* count, cudaStream_t s) {
  export_list_kernel<<<64, 256, 0, s>>>(hdr, items, qb, out, capacity, count);
  return cudaGetLastError();
}

cudaError_t launch_bwd_prep(const PrepParams& p, int sms, cudaStream_t s) {
  bwd_prep_kernel<<<p.n_sched + sms * 2, kSchedThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const FinParams& p, int sms, cudaStream_t s) {
  const long long groups = (static_cast<long long>(p.Lq) * p.H * (p.D / 4) + 31) / 32;
  const int grid = static_cast<int>(std::min<long long>(groups, 8LL * sms));
  finalize_kernel<<<grid > 0 ? grid : 1, kFinThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fill_empty(__nv_bfloat16* out, float* lse, long long rows, int D,
                              cudaStream_t s) {
  fill_empty_kernel<<<256, 256, 0, s>>>(out, lse, rows, D);
  return cudaGetLastError();
}

}  // namespace jfa
