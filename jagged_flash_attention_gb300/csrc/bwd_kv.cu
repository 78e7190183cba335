// Backward, pass 1 of 2: dK and dV for sm_103a (self-attention and
// broadcast-Q).
//
// "Optimizing Jagged Flash Attention with TLX" (pytorch.org), "Scheduling
// jagged tiles across SMs": the dK/dV pass loops over K/V blocks on the
// outside and the query tiles on the inside; items are the valid (sequence,
// head, K/V block) tiles, block-innermost.  For self-attention the dQ part
// of the five products runs in a separate query-outer pass (bwd_q.cu) that
// accumulates dQ on chip, so this pass needs four products per block and no
// global dQ accumulator:
//   S^T  = K Q^T        (SS)                 -> TMEM [0,128)
//   dP^T = V dO^T       (SS)                 -> TMEM [128,256)
//   P^T  = exp2(S^T * scale*log2e - LSE*log2e), bf16 pairs over S^T's columns
//   dS^T = bf16(P^T) * bf16(dP^T - Delta),     bf16 pairs over dP^T's columns
//   dV  += P^T dO       (TS, B = dO MN-major)
//   dK  += dS^T Q       (TS, B = Q MN-major)
// The score math is split into a P part (needs S^T) and a dS part (needs
// dP^T), and the MMAs of consecutive query tiles are interleaved:
//   dV(g), S(g+1), dK(g), dP(g+1), dV(g+1), ...
// so the P part of tile g+1 runs under dK(g) + dP(g+1) and its dS part under
// dV(g+1) + S(g+2).  S(g+1) / dP(g+1) overwrite P^T(g) / dS^T(g) right after
// the dV / dK MMAs that read them (MMAs of one CTA execute in issue order).
//
// CTA = 19 warps: warps 0-15 score/gradient math (warp w: TMEM lanes
// 32*(w%4).. = key rows, query columns 32*(w/4)..; four math warps per SM
// sub-partition, so that each part's TMEM load -> math -> TMEM store chain
// is hidden by the others) and the dK/dV epilogue, warp 16 TMA producer
// (decodes items one ahead, publishes them in shared memory, prefetches the
// next item's first boxes into L2; Q, dO and the row statistics of a stage
// have their own barriers, the statistics freed by the math right after
// their dS part; a Q box a stage still holds is not loaded again; V is
// loaded before the next item is decoded), warp 17 MMA issuer, warp 18 the
// store warp (TMA stores of full dK/dV blocks).
// Variants: with a local mask (causal or a sliding window) a key block
// visits only the query tiles of its band; with GQA an item is a block of
// one K/V head and its query tiles are those of the G query heads that read
// it, so dK and dV sum over the group without leaving the CTA.
// Broadcast-Q ("Optimizing Jagged Flash Attention with TLX", section 1):
// the query tiles of every item are the tiles of the one dense Q, dO is the
// sequence's own [q_len, D] block of the [B, q_len, H, D] tensor (a 4-D
// tensor map zero-fills rows past q_len), and the row statistics come from
// a per-sequence layout padded to whole tiles (padding rows give P = 0).
// Its work list is head-outer, so a CTA's consecutive items usually share
// the dense-Q tiles its stages hold.
// At an item boundary the math warps compute the next item's first P part,
// then the item's dV epilogue, the next item's first dS part, and only then
// the item's dK epilogue, so that the first products of the next item wait
// for one TMEM load each rather than for the epilogue.
//
// PAIR ("Optimizing Jagged Flash Attention with TLX", "2-CTA collaborative
// MMA (backward)"): a cluster of two CTAs takes two adjacent key blocks of
// one (sequence, head), CTA r block 2j + r, and the pair's products are
// cta_group::2 products with M = 256 (the two key blocks) issued by CTA 0:
// each CTA keeps its key block's K, V and accumulators and holds half of
// every B operand.  Per query tile CTA r loads query rows [64r, 64r + 64) of
// Q and dO with all head-dim columns (the N half of S^T and dP^T) and all
// 128 rows of head-dim columns [64r, 64r + 64) (the N half of dK and dV):
// [rows-half slab 0 | rows-half slab 1 | columns-half slab], 32 KB like the
// single-CTA stage.  Both CTAs' loads complete on CTA 0's full barriers
// (CTA 0 expects both CTAs' bytes), the commits arrive on both CTAs'
// barriers, and each CTA's math warps report P^T / dS^T and the freed
// accumulators to CTA 0's issuer, one arrive per warp.  Items are the key
// block pairs of the work list, taken by the pairs in a fixed stride (both
// CTAs walk the same items without exchanging tickets).  Self-attention
// without a local mask and broadcast-Q, D = 128.
#include "common.cuh"
#include "ptx.cuh"

namespace jfa {
namespace {

constexpr int kMathWarps = 16;
constexpr int kMath = 32 * kMathWarps;
constexpr int kProducerWarp = kMathWarps;
constexpr int kMmaWarp = kMathWarps + 1;
constexpr int kStoreWarp = kMathWarps + 2;
constexpr int kThreads = 32 * (kMathWarps + 3);

template <int D>
struct KvCfg {
  static constexpr int NSQ = 2;              // Q / dO ring depth
  static constexpr int kTile = kBM * D * 2;  // bytes of a 128-row bf16 tile
  static constexpr int kSlabs = D / 64;
  // Two K buffers (the next item's K is loaded while this item runs), one V
  // buffer (released once the item's last dP^T has read it).
  static constexpr int kK = 0;
  static constexpr int kV = 2 * kTile;
  static constexpr int kQ = 3 * kTile;
  static constexpr int kDO = kQ + NSQ * kTile;
  // {-LSE*log2e, -Delta} of the 128 query rows of each Q / dO stage
  static constexpr int kStatBytes = kBM * 8;
  static constexpr int kStat = kDO + NSQ * kTile;
  static constexpr int kCtl = kStat + NSQ * kStatBytes;
  static constexpr int kSmem = kCtl + 512;
  static constexpr uint32_t kColS = 0, kColDP = 128;
  static constexpr uint32_t kColDV = 256, kColDK = 256 + D;
};

struct RowBox {
  int row, shift, n;  // TMA row coordinate, rows moved back, valid rows
};
__device__ __forceinline__ RowBox row_box(int start, int remaining, int T) {
  RowBox r;
  r.shift = max(0, start + 128 - T);
  r.row = start - r.shift;
  r.n = min(128, remaining);
  return r;
}

// With GQA an item is a block of one K/V head, and its query tiles are the
// tiles [t0, t0 + ntq) of each of the G query heads that read that K/V head,
// head-major: tile i is query tile t0 + i % ntq of query head h * G + i / ntq.
struct KvItem {
  int b, h, kb;  // sequence, K/V head, key block
  int off0, L;
  RowBox kt;        // keys of this block
  int t0, ntq, nt;  // first query tile, tiles per query head, nt = G * ntq
};

// One staged output tensor for the store warp: which = 0: dV, 1: dK, -1:
// no more; buf: byte offset of the staging buffer in shared memory.
struct StoreJob {
  int which, buf, h, row, kbuf;
};

struct KvCtl {
  uint64_t k_full[2], k_empty[2], v_full, v_empty;
  // Query-tile ring: Q (with the rows' statistics) and dO of a stage have
  // their own barriers: Q is read by S^T and dK, dO by dP^T and dV.  The
  // full barriers are per 64-column slab ([stage][slab]; the statistics
  // ride with slab 0), so that a product's first K steps need only slab 0.
  uint64_t q_full[2][2], q_empty[2], do_full[2][2], do_empty[2];
  // Row statistics of a stage: loaded as soon as the math's dS part of the
  // stage's previous tile has read them (before its Q is free), so that a Q
  // box a stage already holds needs no copy on the issuer's path.
  uint64_t stat_full[2], stat_empty[2];
  uint64_t s_full, dp_full, p_full, ds_full;
  uint64_t dkdv_full, dv_empty, dk_empty;
  uint64_t epi;  // math-warp sync of the staged epilogue stores
  // Staged tensor -> store warp, one barrier per job slot (a slot's next
  // phase can complete only after the store warp has taken its job); dV's
  // rows read by the store.
  uint64_t stg_full[2], stg_empty;
  StoreJob job[2];               // what the store warp stores, by submission
  uint64_t item_full[2], item_empty[2];
  uint64_t drain;
  KvItem item[2];  // decoded by the producer; b < 0: no more items
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

// TMEM column of the bf16 pairs of queries 16k..16k+15 in a packed P^T /
// dS^T: query quarter q = k/2 (columns 32q..32q+31 of the fp32 tile) keeps
// its 16 packed columns at 32q.
__device__ __forceinline__ uint32_t pack_col(int k) { return 32 * (k >> 1) + 8 * (k & 1); }


template <bool LOCAL, bool BCAST, bool PAIR>
__device__ __forceinline__ KvItem decode(const BwdParams& p, int idx, int T, int rank) {
  KvItem f;
  const Item it = p.items[idx];
  f.b = it.x;
  f.h = it.y >> 16;
  // a pair item is a pair of key blocks; CTA r of the pair takes block 2j + r
  // (past the sequence for the second CTA of an odd count: nothing stored)
  f.kb = PAIR ? 2 * (it.y & 0xffff) + rank : it.y & 0xffff;
  f.off0 = p.offsets[f.b];
  f.L = p.offsets[f.b + 1] - f.off0;
  f.kt = row_box(f.off0 + f.kb * kBN, f.L - f.kb * kBN, T);
  if (BCAST) {
    f.t0 = 0;
    f.ntq = cdiv(p.Lq, kBM);
  } else if (LOCAL) {  // the query tiles that admit a key of the block
    const int ka = f.kb * kBN;
    query_tiles(ka, ka + f.kt.n - 1, f.L, p.wl, p.wr, &f.t0, &f.ntq);
  } else {
    f.t0 = 0;
    f.ntq = cdiv(f.L, kBM);
  }
  f.nt = p.G * f.ntq;
  return f;
}

// Query head and query tile of tile i of item f.
__device__ __forceinline__ int q_head(const BwdParams& p, const KvItem& f, int i) {
  return f.h * p.G + i / f.ntq;
}
__device__ __forceinline__ int q_tile(const KvItem& f, int i) { return f.t0 + i % f.ntq; }

// Query tile t of item f: self-attention, rows of the sequence (moved back so
// the box never reads past row T); broadcast, rows of the dense Q.
template <bool BCAST>
__device__ __forceinline__ RowBox q_box(const BwdParams& p, const KvItem& f, int t, int T) {
  if (BCAST) {
    RowBox r;
    r.row = t * kBM;
    r.shift = 0;
    r.n = min(kBM, p.Lq - t * kBM);
    return r;
  }
  return row_box(f.off0 + t * kBM, f.L - t * kBM, T);
}

// Statistics of the 128 rows of query tile t of query head qh (1 KB,
// 32-byte aligned): self,
// the copy in which the box's first row starts a group; broadcast, the
// sequence's rows in the layout padded to whole tiles.
template <bool BCAST>
__device__ __forceinline__ const float* stat_src(const BwdParams& p, const KvItem& f, int qh,
                                                 const RowBox& qb, int t, int T) {
  if (BCAST) {
    const long long lq_pad = static_cast<long long>(cdiv(p.Lq, kBM)) * kBM;
    return p.stat + stat_float((static_cast<long long>(f.b) * p.H + qh) * lq_pad + t * kBM);
  }
  const long long sidx = static_cast<long long>(qh) * T + qb.row;
  const int sk = static_cast<int>((sidx + kStatPad) & 3);
  return p.stat + sk * p.stat_stride + stat_float(stat_pos(sidx, sk));
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, int* err) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > JFA_WAIT_LIMIT_CYCLES) {
      atomicOr(err, kErrTimeout);
      return;
    }
  }
}

// Next work item of the CTA as the producer decoded it (called by whole
// warps: the math warps and the MMA warp).  False when the list is done or a
// wait gave up (then *ok is false too).
__device__ __forceinline__ bool next_item(KvCtl* c, uint32_t n, KvItem* f, bool* ok, int* err,
                                          bool release = true) {
  const int slot = n & 1;
  if (!mbar_wait_warp(&c->item_full[slot], (n >> 1) & 1, &c->abort, err)) {
    *ok = false;
    return false;
  }
  *f = c->item[slot];
  __syncwarp();
  if (release && (threadIdx.x & 31) == 0) mbar_arrive(&c->item_empty[slot]);
  return f->b >= 0;
}

template <int D, bool LOCAL, bool BCAST, bool PAIR>
__device__ void producer_role(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                              const CUtensorMap* tdo, const CUtensorMap* tq_h,
                              const CUtensorMap* tdo_h, const BwdParams& p, uint8_t* smem,
                              KvCtl* c) {
  using C = KvCfg<D>;
  const int n_items = p.hdr->n_items;
  const int T = p.hdr->T;
  const int rank = PAIR ? static_cast<int>(cluster_rank()) : 0;
  const bool lead = rank == 0;
  // Items: the shared ticket; a pair walks the list in a fixed stride.
  uint32_t ki = 0;
  auto take = [&]() -> int {
    if (PAIR) return static_cast<int>((blockIdx.x >> 1) + (ki++) * (gridDim.x >> 1));
    return atomicAdd(&p.hdr->ticket, 1);
  };
  // A pair's loads complete on CTA 0's barriers, which expect both CTAs'
  // bytes; CTA 1 only issues its copies.
  auto expect = [&](uint64_t* bar, uint32_t bytes) {
    if (!PAIR)
      mbar_arrive_expect_tx(bar, bytes);
    else if (lead)
      mbar_arrive_expect_tx(bar, 2 * bytes);
  };
  auto load3 = [&](void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1, int c2) {
    if (PAIR && !lead)
      tma_load_3d_pair(dst, m, smem_in_cta(bar, 0), c0, c1, c2);
    else
      tma_load_3d(dst, m, bar, c0, c1, c2);
  };
  auto load4 = [&](void* dst, const CUtensorMap* m, uint64_t* bar, int c0, int c1, int c2, int c3) {
    if (PAIR && !lead)
      tma_load_4d_pair(dst, m, smem_in_cta(bar, 0), c0, c1, c2, c3);
    else
      tma_load_4d(dst, m, bar, c0, c1, c2, c3);
  };
  // Q or dO tile of query head qh at box row `row` into ring stage `st` of
  // buffer `buf`, slab barriers full[0..1]; dO of broadcast-Q is the 4-D
  // [B, q_len, H, D] tensor (coordinate b), everything else 3-D.
  auto load_tile = [&](int buf, int st, const CUtensorMap* m, const CUtensorMap* m_h,
                       uint64_t* full, int qh, int row, int b, bool four_d) {
    uint8_t* dst = smem + buf + st * C::kTile;
    if (!PAIR) {
#pragma unroll
      for (int s = 0; s < C::kSlabs; ++s) {
        mbar_arrive_expect_tx(&full[s], 16384);
        if (four_d)
          tma_load_4d(dst + s * 16384, m, &full[s], s * 64, qh, row, b);
        else
          tma_load_3d(dst + s * 16384, m, &full[s], s * 64, qh, row);
      }
      return;
    }
    // [rows-half slab 0 | rows-half slab 1 | columns-half]: slab 0 of the
    // row half on barrier 0, the rest on barrier 1
    expect(&full[0], 8192);
    expect(&full[1], 8192 + 16384);
    if (four_d) {
      load4(dst, m_h, &full[0], 0, qh, row + 64 * rank, b);
      load4(dst + 8192, m_h, &full[1], 64, qh, row + 64 * rank, b);
      load4(dst + 16384, m, &full[1], 64 * rank, qh, row, b);
    } else {
      load3(dst, m_h, &full[0], 0, qh, row + 64 * rank);
      load3(dst + 8192, m_h, &full[1], 64, qh, row + 64 * rank);
      load3(dst + 16384, m, &full[1], 64 * rank, qh, row);
    }
  };
  // gdo / gst: stages whose dO / statistics copy was issued
  uint32_t it = 0, gq = 0, gdo = 0, gst = 0, nk = 0, nv = 0;
  bool ok = true;
  // Q box each ring stage holds (query head, row; -1: none).  When the next
  // tile of a stage is the same box (broadcast: consecutive items of one head
  // walk the same dense-Q tiles) it is not loaded again; only its row
  // statistics are.  Nothing but these loads writes a Q stage.
  static_assert(C::NSQ == 2, "held boxes: two stages");
  long long held0 = -1, held1 = -1;
  // One-item lookahead: the next item is taken and decoded while this one's
  // loads go out, and its K, V and first Q / dO boxes are prefetched into
  // L2, so that at the item boundary they come from L2 rather than HBM.
  auto fetch = [&](KvItem& f) {
    const int idx = take();
    if (idx < n_items)
      f = decode<LOCAL, BCAST, PAIR>(p, idx, T, rank);
    else
      f.b = -1;
  };
  auto prefetch = [&](const KvItem& f) {
    const RowBox qb = q_box<BCAST>(p, f, f.t0, T);
    const int qh = f.h * p.G;  // the first tile's query head
#pragma unroll
    for (int s = 0; s < C::kSlabs; ++s) {
      if (f.kt.row >= 0) {
        tma_prefetch_l2_3d(tk, s * 64, f.h, f.kt.row);
        tma_prefetch_l2_3d(tv, s * 64, f.h, f.kt.row);
      }
      if (BCAST) {  // the dense Q stays in L2; the sequence's dO
        tma_prefetch_l2_4d(tdo, s * 64, qh, 0, f.b);
      } else if (qb.row >= 0) {
        tma_prefetch_l2_3d(tq, s * 64, qh, qb.row);
        tma_prefetch_l2_3d(tdo, s * 64, qh, qb.row);
      }
    }
  };
  KvItem f;
  fetch(f);
  for (uint32_t n = 0; ok; ++n) {
    const int slot = n & 1;
    if (!mbar_wait(&c->item_empty[slot], ((n >> 1) & 1) ^ 1, &c->abort, p.err)) break;
    c->item[slot] = f;
    mbar_arrive(&c->item_full[slot]);
    if (f.b < 0) break;
    KvItem nx;
    nx.b = -1;
    // Order of the item's loads: K, the first Q / dO, V (V waits for the
    // previous item's last dP^T), then the other Q / dO tiles.
    const int ks = it & 1;
    if (!mbar_wait(&c->k_empty[ks], ((it >> 1) & 1) ^ 1, &c->abort, p.err)) break;
    expect(&c->k_full[ks], C::kTile);
#pragma unroll
    for (int s = 0; s < C::kSlabs; ++s)
      load3(smem + C::kK + ks * C::kTile + s * 16384, tk, &c->k_full[ks], s * 64, f.h, f.kt.row);
    ++nk;
    for (int i = 0; i < f.nt; ++i) {
      const uint32_t g = gq;
      const int st = g % C::NSQ;
      // dO first: its stage frees after dV, a product before Q's (after dK),
      // so that its bytes are in by the time Q's load starts, and Q, which
      // S^T(g) waits for, has the L2 path to itself.
      if (!mbar_wait(&c->do_empty[st], ((g / C::NSQ) & 1) ^ 1, &c->abort, p.err)) {
        ok = false;
        break;
      }
      const int t = q_tile(f, i), qh = q_head(p, f, i);
      const RowBox qb = q_box<BCAST>(p, f, t, T);
      load_tile(C::kDO, st, tdo, tdo_h, c->do_full[st], qh, qb.row, f.b, BCAST);
      ++gdo;  // counted now: a wait below that gives up must not hide these copies from the drain
      // Row statistics of the box: 32 whole groups (1 KB).
      if (!mbar_wait(&c->stat_empty[st], ((g / C::NSQ) & 1) ^ 1, &c->abort, p.err)) {
        ok = false;
        break;
      }
      mbar_arrive_expect_tx(&c->stat_full[st], C::kStatBytes);
      bulk_load(smem + C::kStat + st * C::kStatBytes, stat_src<BCAST>(p, f, qh, qb, t, T),
                C::kStatBytes, &c->stat_full[st]);
      ++gst;
      if (!mbar_wait(&c->q_empty[st], ((g / C::NSQ) & 1) ^ 1, &c->abort, p.err)) {
        ok = false;
        break;
      }
      const long long tag = (static_cast<long long>(qh) << 32) | static_cast<uint32_t>(qb.row);
      const bool reuse = (st == 0 ? held0 : held1) == tag;
      if (st == 0)
        held0 = tag;
      else
        held1 = tag;
      if (reuse) {  // Q already in the stage: the phases complete at once
        if (!PAIR || lead) {
#pragma unroll
          for (int s = 0; s < C::kSlabs; ++s) mbar_arrive(&c->q_full[st][s]);
        }
      } else {
        load_tile(C::kQ, st, tq, tq_h, c->q_full[st], qh, qb.row, f.b, false);
      }
      ++gq;
      if (i == 0) {
        // V first: the item's first dP^T waits for it.  The next item's
        // ticket is taken before the wait and decoded (two dependent global
        // loads) only once V's copy is out.
        const int nidx = take();
        if (!mbar_wait(&c->v_empty, (it & 1) ^ 1, &c->abort, p.err)) {
          ok = false;
          break;
        }
        expect(&c->v_full, C::kTile);
#pragma unroll
        for (int s = 0; s < C::kSlabs; ++s)
          load3(smem + C::kV + s * 16384, tv, &c->v_full, s * 64, f.h, f.kt.row);
        ++nv;
        if (nidx < n_items) {
          nx = decode<LOCAL, BCAST, PAIR>(p, nidx, T, rank);
          prefetch(nx);
        }
      }
    }
    ++it;
    f = nx;
  }
  // A pair's copies complete on CTA 0's barriers: CTA 0 drains both CTAs'
  // (the pair's closing cluster barrier keeps CTA 1 until then).
  if (!PAIR || lead) {
    for (uint32_t j = nk > 2 ? nk - 2 : 0; j < nk; ++j)
      drain_wait(&c->k_full[j & 1], (j >> 1) & 1, p.err);
    if (nv > 0) drain_wait(&c->v_full, (nv - 1) & 1, p.err);
    for (uint32_t g = gq > C::NSQ ? gq - C::NSQ : 0; g < gq; ++g)
#pragma unroll
      for (int s = 0; s < C::kSlabs; ++s)
        drain_wait(&c->q_full[g % C::NSQ][s], (g / C::NSQ) & 1, p.err);
    for (uint32_t g = gdo > C::NSQ ? gdo - C::NSQ : 0; g < gdo; ++g)
#pragma unroll
      for (int s = 0; s < C::kSlabs; ++s)
        drain_wait(&c->do_full[g % C::NSQ][s], (g / C::NSQ) & 1, p.err);
  }
  for (uint32_t g = gst > C::NSQ ? gst - C::NSQ : 0; g < gst; ++g)
    drain_wait(&c->stat_full[g % C::NSQ], (g / C::NSQ) & 1, p.err);
}

template <int D, bool LOCAL, bool PAIR>
__device__ void mma_role(const BwdParams& p, uint8_t* smem, KvCtl* c, uint32_t tbase) {
  using C = KvCfg<D>;
  // Run by the whole warp; the elected lane issues products and commits.
  // PAIR: run by CTA 0 only; M = 256 covers both CTAs' key blocks.
  const uint32_t leader = elect_one();
  constexpr int kM = PAIR ? 256 : 128;
  const uint32_t id_st = idesc_bf16_f32(kM, 128, false, false);  // S^T, dP^T
  const uint32_t id_kv = idesc_bf16_f32(kM, D, false, true);     // dV, dK (A in TMEM)
  // Offsets in a query-tile stage: single CTA, 64-column slab k at 16 KB k;
  // pair, the row half's slab k at 8 KB k and the column half at 16 KB.
  constexpr uint32_t kSlabN = PAIR ? 8192 : 16384, kColsM = PAIR ? 16384 : 0;
  auto ss = [&](uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
    if (PAIR)
      mma_ss_pair(d, a, b, id, acc);
    else
      mma_ss(d, a, b, id, acc);
  };
  auto ts = [&](uint32_t d, uint32_t a, uint64_t b, uint32_t id, uint32_t acc) {
    if (PAIR)
      mma_ts_pair(d, a, b, id, acc);
    else
      mma_ts(d, a, b, id, acc);
  };
  auto commit = [&](uint64_t* bar) {
    if (!leader) return;
    if (PAIR)
      mma_commit_pair(bar);
    else
      mma_commit(bar);
  };
  // Barriers the math warps arrive on (both CTAs' warps for a pair).
  auto wait_math = [&](uint64_t* bar, uint32_t parity) {
    return mbar_wait_warp(bar, parity, &c->abort, p.err);
  };
  // Descriptors built once; per tile and K step only adds remain.
  const uint64_t dk_k0 = smem_desc_sw128(smem_addr(smem + C::kK), 16, 1024);
  const uint64_t dv_k = smem_desc_sw128(smem_addr(smem + C::kV), 16, 1024);
  const uint64_t dq_k0 = smem_desc_sw128(smem_addr(smem + C::kQ), 16, 1024);
  const uint64_t ddo_k0 = smem_desc_sw128(smem_addr(smem + C::kDO), 16, 1024);
  const uint64_t dq_m0 = smem_desc_sw128(smem_addr(smem + C::kQ), 16384, 1024);
  const uint64_t ddo_m0 = smem_desc_sw128(smem_addr(smem + C::kDO), 16384, 1024);
  const uint32_t tS = tbase + C::kColS, tDP = tbase + C::kColDP;
  const uint32_t tDV = tbase + C::kColDV, tDK = tbase + C::kColDK;
  // Slab s of the query tile of ring index g (Q or dO), before its first K step.
  auto wait_slab = [&](uint64_t (*full)[2], uint32_t g, int s) {
    return mbar_wait_warp(&full[g % C::NSQ][s], (g / C::NSQ) & 1, &c->abort, p.err);
  };
  // S^T(g) and dP^T(g): K steps 4k.. read 64-column slab k of Q / dO; the
  // issuer waits for slab 0 before the product (wait_q / wait_do) and for
  // slab 1 between its K steps 3 and 4.
  auto issue_s = [&](uint32_t g, uint64_t dk_k) {
    const uint64_t dq_k = desc_add(dq_k0, (g % C::NSQ) * C::kTile);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      if (k > 0 && k % 4 == 0) {
        if (!wait_slab(c->q_full, g, k / 4)) return false;
        tc_fence_after();
      }
      const uint32_t off_a = (k / 4) * 16384 + (k % 4) * 32;
      const uint32_t off_b = (k / 4) * kSlabN + (k % 4) * 32;
      if (leader) ss(tS, desc_add(dk_k, off_a), desc_add(dq_k, off_b), id_st, k > 0);
    }
    return true;
  };
  auto issue_dp = [&](uint32_t g) {
    const uint64_t ddo_k = desc_add(ddo_k0, (g % C::NSQ) * C::kTile);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      if (k > 0 && k % 4 == 0) {
        if (!wait_slab(c->do_full, g, k / 4)) return false;
        tc_fence_after();
      }
      const uint32_t off_a = (k / 4) * 16384 + (k % 4) * 32;
      const uint32_t off_b = (k / 4) * kSlabN + (k % 4) * 32;
      if (leader) ss(tDP, desc_add(dv_k, off_a), desc_add(ddo_k, off_b), id_st, k > 0);
    }
    return true;
  };
  // A operand column of query block k (16 queries): the packed P^T / dS^T
  // of query quarter k/2 starts at its own first column, 32 * (k/2).
  auto issue_dv = [&](uint32_t g, bool acc) {
    const uint64_t ddo_m = desc_add(ddo_m0, (g % C::NSQ) * C::kTile);
#pragma unroll
    for (int k = 0; k < kBM / 16; ++k)
      if (leader) ts(tDV, tS + pack_col(k), desc_add(ddo_m, kColsM + k * 2048), id_kv, acc || (k > 0));
  };
  auto issue_dk = [&](uint32_t g, bool acc) {
    const uint64_t dq_m = desc_add(dq_m0, (g % C::NSQ) * C::kTile);
#pragma unroll
    for (int k = 0; k < kBM / 16; ++k)
      if (leader) ts(tDK, tDP + pack_col(k), desc_add(dq_m, kColsM + k * 2048), id_kv, acc || (k > 0));
  };
  auto wait_q = [&](uint32_t g) { return wait_slab(c->q_full, g, 0); };
  auto wait_do = [&](uint32_t g) { return wait_slab(c->do_full, g, 0); };
  auto wait_p = [&](uint32_t g) { return wait_math(&c->p_full, g & 1); };
  auto wait_ds = [&](uint32_t g) { return wait_math(&c->ds_full, g & 1); };
  uint32_t it = 0, gq = 0;
  bool ok = true, issued = false;
  for (uint32_t n = 0; ok; ++n) {
    KvItem f;
    if (!next_item(c, n, &f, &ok, p.err)) break;
    const int ks = it & 1;
    if (!mbar_wait_warp(&c->k_full[ks], (it >> 1) & 1, &c->abort, p.err)) break;
    const uint64_t dk_k = desc_add(dk_k0, ks * C::kTile);
    const uint32_t g0 = gq;
    if (!wait_q(g0)) break;
    tc_fence_after();
    issued = true;
    if (!issue_s(g0, dk_k)) break;
    commit(&c->s_full);
    // V is released after the item's last dP^T; K after the item epilogue,
    // which stages its stores in the K buffer.
    if (!mbar_wait_warp(&c->v_full, it & 1, &c->abort, p.err)) break;
    if (!wait_do(g0)) break;
    tc_fence_after();
    if (!issue_dp(g0)) break;
    commit(&c->dp_full);
    if (f.nt == 1) commit(&c->v_empty);
    // dV(g0) restarts the accumulator the previous item's epilogue reads
    // (dK(g0) waits below for the dK one).
    if (!wait_math(&c->dv_empty, (it & 1) ^ 1)) break;
    // Order per tile g: dV(g), S(g+1), dK(g), dP(g+1).  Every product is
    // committed whole, and the issuer waits only before a product that reads
    // what the math produced (P^T before dV, dS^T before dK) or for the query
    // tile's slabs that S(g+1) and dP(g+1) read (slab 1 between their K
    // steps 3 and 4, so that the first half runs while it lands).
    // S(g+1) / dP(g+1) overwrite P^T(g) / dS^T(g) after dV(g) / dK(g),
    // which were issued before them.
    for (int i = 0; i < f.nt; ++i) {
      const uint32_t g = g0 + i;
      const bool more = i + 1 < f.nt;
      if (!wait_p(g)) { ok = false; break; }
      tc_fence_after();
      issue_dv(g, i > 0);
      commit(&c->do_empty[g % C::NSQ]);
      if (more) {
        if (!wait_q(g + 1)) { ok = false; break; }
        tc_fence_after();
        if (!issue_s(g + 1, dk_k)) { ok = false; break; }
        commit(&c->s_full);
      }
      if (!wait_ds(g)) { ok = false; break; }
      if (i == 0 && !wait_math(&c->dk_empty, (it & 1) ^ 1)) { ok = false; break; }
      tc_fence_after();
      issue_dk(g, i > 0);
      commit(&c->q_empty[g % C::NSQ]);
      if (more) {
        if (!wait_do(g + 1)) { ok = false; break; }
        tc_fence_after();
        if (!issue_dp(g + 1)) { ok = false; break; }
        commit(&c->dp_full);
        if (i + 2 == f.nt) commit(&c->v_empty);
      }
    }
    if (!ok) break;
    gq += f.nt;
    commit(&c->dkdv_full);
    ++it;
  }
  if (issued && leader) {
    commit(&c->drain);
    drain_wait(&c->drain, 0, p.err);
  }
}

template <int D, bool LOCAL, bool BCAST, bool PAIR>
__device__ void math_role(const BwdParams& p, uint8_t* smem, KvCtl* c, uint32_t tbase) {
  using C = KvCfg<D>;
  // What the issuer waits for (P^T, dS^T, a freed accumulator): every
  // thread arrives; in a pair one arrive per warp of either CTA on CTA 0's
  // barrier, CTA 1's from across the pair (the warp's TMEM accesses are
  // complete and fenced before it).
  const bool remote = PAIR && cluster_rank() != 0;
  auto to_issuer = [&](uint64_t* bar) {
    if (!PAIR) {
      mbar_arrive(bar);
      return;
    }
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
      if (remote)
        mbar_arrive_remote(smem_in_cta(bar, 0));
      else
        mbar_arrive(bar);
    }
  };
  const int r = threadIdx.x & 127;    // TMEM lane = key row of the block
  const int qd = threadIdx.x >> 7;    // query columns [32*qd, 32*qd + 32)
  const int cbase = 32 * qd;
  const uint32_t lane_base = static_cast<uint32_t>((r >> 5) * 32) << 16;
  const int T = p.hdr->T;
  const float sl2 = p.scale_log2;
  const uint64_t sl2x2 = f2_pack(sl2, sl2);
  // Statistics of columns 4j..4j+3 of tile g: -LSE*log2e at st4[2j], -Delta
  // at st4[2j + 1]; they arrive with slab 0 of the tile's Q stage.
  auto stats = [&](uint32_t g) {
    return reinterpret_cast<const float4*>(smem + C::kStat + (g % C::NSQ) * C::kStatBytes);
  };
  // ---- P part of tile i (ring index g) of item f: P^T = exp2(S^T *
  // scale*log2e - LSE*log2e), kept as bf16 pairs of this thread's 32 columns.
  auto p_part = [&](const KvItem& f, int i, uint32_t g, uint32_t (&pk)[16]) {
    const int key = f.kb * kBN - f.kt.shift + r;  // local key index of this lane
    const int t = q_tile(f, i);
    const RowBox qb = q_box<BCAST>(p, f, t, T);
    const int q0 = t * kBM - qb.shift;  // local query index of column 0
    if (!mbar_wait_warp(&c->stat_full[g % C::NSQ], (g / C::NSQ) & 1, &c->abort, p.err)) return false;
    const float4* st4 = stats(g);
    // Admissible query columns [lo, hi): the box's rows of the sequence
    // and, with a local mask, the queries in [key - wr, key + wl].
    int lo = qb.shift, hi = qb.shift + qb.n;
    if (LOCAL) {
      lo = max(lo, key - p.wr - q0);
      hi = min(hi, key + p.wl - q0 + 1);
    }
    const bool ragged = qb.shift > 0 || qb.n < kBM;
    const bool mask = ragged || (LOCAL && __any_sync(0xffffffffu, lo > cbase || hi < cbase + 32));
    const uint32_t span = hi > lo ? static_cast<uint32_t>(hi - lo) : 0u;
    if (!mbar_wait_warp(&c->s_full, g & 1, &c->abort, p.err)) return false;
    tc_fence_after();
    {
      uint32_t sraw[32];
      tmem_ld32(tbase + lane_base + C::kColS + cbase, sraw);
      tmem_wait_ld();
      // Rows of keys outside the sequence are left unmasked: row r of dV
      // and dK depends only on row r of P^T and dS^T, and those rows are
      // never stored.
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 nl = st4[2 * (cbase / 4 + j)];
        const float2 x01 = f2_unpack(ffma2(
            f2_pack(__uint_as_float(sraw[4 * j]), __uint_as_float(sraw[4 * j + 1])), sl2x2,
            f2_pack(nl.x, nl.y)));
        const float2 x23 = f2_unpack(ffma2(
            f2_pack(__uint_as_float(sraw[4 * j + 2]), __uint_as_float(sraw[4 * j + 3])), sl2x2,
            f2_pack(nl.z, nl.w)));
        pk[2 * j] = pack_bf16x2(ex2_approx(x01.x), ex2_approx(x01.y));
        pk[2 * j + 1] = pack_bf16x2(ex2_approx(x23.x), ex2_approx(x23.y));
      }
      if (mask) {  // ragged tile, or one a band edge crosses: zero inadmissible columns
#pragma unroll
        for (int i2 = 0; i2 < 16; ++i2) {
          const int col = cbase + 2 * i2;
          pk[i2] &= (static_cast<uint32_t>(col - lo) < span ? 0x0000ffffu : 0u) |
                    (static_cast<uint32_t>(col + 1 - lo) < span ? 0xffff0000u : 0u);
        }
      }
      // bf16 pairs of this quarter's columns land in its own first 16
      // columns, already read above.
      tmem_st16(tbase + lane_base + C::kColS + cbase, pk);
    }
    tmem_wait_st();
    tc_fence_before();
    to_issuer(&c->p_full);
    return true;
  };
  // ---- dS part of tile g: dS^T = P^T (dP^T - Delta): the difference in
  // fp32, rounded to bf16, times the bf16 P.
  auto ds_part = [&](uint32_t g, const uint32_t (&pk)[16]) {
    const float4* st4 = stats(g);
    if (!mbar_wait_warp(&c->dp_full, g & 1, &c->abort, p.err)) return false;
    tc_fence_after();
    {
      uint32_t praw[32];
      tmem_ld32(tbase + lane_base + C::kColDP + cbase, praw);
      tmem_wait_ld();
      uint32_t w[16];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 nd = st4[2 * (cbase / 4 + j) + 1];
        const float2 d01 = f2_unpack(fadd2(
            f2_pack(__uint_as_float(praw[4 * j]), __uint_as_float(praw[4 * j + 1])),
            f2_pack(nd.x, nd.y)));
        const float2 d23 = f2_unpack(fadd2(
            f2_pack(__uint_as_float(praw[4 * j + 2]), __uint_as_float(praw[4 * j + 3])),
            f2_pack(nd.z, nd.w)));
        w[2 * j] = bmul2(pk[2 * j], pack_bf16x2(d01.x, d01.y));
        w[2 * j + 1] = bmul2(pk[2 * j + 1], pack_bf16x2(d23.x, d23.y));
      }
      tmem_st16(tbase + lane_base + C::kColDP + cbase, w);
    }
    tmem_wait_st();
    tc_fence_before();
    to_issuer(&c->ds_full);
    // this warp's reads of the stage's statistics are done
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&c->stat_empty[g % C::NSQ]);
    return true;
  };
  uint32_t it = 0, gq = 0, ep = 0;
  // Sync of the 512 math threads (bounded mbarrier phases), around the
  // staging of a ragged block's epilogue.
  auto epi_sync = [&]() {
    mbar_arrive(&c->epi);
    const bool r_ = mbar_wait_warp(&c->epi, ep & 1, &c->abort, p.err);
    ++ep;
    return r_;
  };
  // This thread's 32 head-dim columns of dV or dK: D = 128: quarter qd holds
  // columns 32*qd.. of both; D = 64: quarters 0-1 hold dV, 2-3 dK.
  const int dbase = D == 128 ? 32 * qd : 32 * (qd & 1);
  const bool has_dv = D == 128 || qd < 2, has_dk = D == 128 || qd >= 2;
  // One tensor of the item epilogue (which = 0: dV, 1: scale * dK): the
  // accumulator leaves TMEM and is released at once (the next item's first
  // product into it then waits only for this load), then goes through the
  // item's K buffer.  A full key block (all 128 rows in the sequence) is
  // staged in the 128-byte-swizzled layout of the output tensor map (slab s
  // of 64 columns at s*16 KB, row r at r*128 bytes, 16-byte chunk c at
  // c ^ (r mod 8)) and handed to the store warp, which stores it by TMA:
  // the math warps wait neither for the stores nor for the store warp,
  // except, before staging dK, for dV's store to have read the buffer.  The
  // rows of a ragged block are stored by the math warps, whole rows per
  // warp store (one thread holds 64 bytes of one key row, 2 KB from the next
  // row's; stored directly, every warp store would touch 32 lines), from the
  // layout row r at 2*D bytes, 16-byte chunk c at c ^ (r mod D/8)
  // (conflict-free both ways).
  // Tensors handed to the store warp: full blocks hand over dV, dK, dV, ...,
  // so dK is always the odd one and its dV the (ns >> 1)-th dV.
  uint32_t ns = 0;
  auto epi_tensor = [&](const KvItem& f, uint32_t itf, int which, bool full) {
    uint8_t* stg = smem + C::kK + (itf & 1) * C::kTile;
    const bool mine = which == 0 ? has_dv : has_dk;
    uint32_t w16[16];
    if (mine) {
      uint32_t a[32];
      tmem_ld32(tbase + lane_base + (which == 0 ? C::kColDV : C::kColDK) + dbase, a);
      tmem_wait_ld();
      const float mul = which == 0 ? 1.f : p.scale;
#pragma unroll
      for (int i2 = 0; i2 < 16; ++i2)
        w16[i2] = pack_bf16x2(__uint_as_float(a[2 * i2]) * mul, __uint_as_float(a[2 * i2 + 1]) * mul);
    }
    tc_fence_before();
    to_issuer(which == 0 ? &c->dv_empty : &c->dk_empty);
    constexpr int kCpr = D / 8;       // 16-byte chunks per row
    constexpr int kRpi = 32 / kCpr;   // rows per warp store
    if (which == 1) {  // dV's rows have left the buffer
      if (full) {
        if (!mbar_wait_warp(&c->stg_empty, (ns >> 1) & 1, &c->abort, p.err)) return false;
      } else if (!epi_sync()) {
        return false;
      }
    }
    if (mine) {
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const uint4 v4 = make_uint4(w16[4 * q4], w16[4 * q4 + 1], w16[4 * q4 + 2], w16[4 * q4 + 3]);
        if (full) {
          const int ch = (dbase % 64) / 8 + q4;
          *reinterpret_cast<uint4*>(stg + (dbase / 64) * 16384 + r * 128 + ((ch ^ (r & 7)) * 16)) = v4;
        } else {
          const int ch = dbase / 8 + q4;
          *reinterpret_cast<uint4*>(stg + r * (2 * D) + ((ch ^ (r & (kCpr - 1))) * 16)) = v4;
        }
      }
    }
    if (full) {
      if (threadIdx.x == 0) {
        StoreJob& j = c->job[ns & 1];
        j.which = which;
        j.buf = C::kK + (itf & 1) * C::kTile;
        j.h = f.h;
        j.row = f.kt.row;
        j.kbuf = itf & 1;
      }
      fence_proxy_async_smem();  // the staged rows, for the TMA store
      mbar_arrive(&c->stg_full[ns & 1]);
      ++ns;
      return true;
    }
    if (!epi_sync()) return false;  // the tensor is staged
    __nv_bfloat16* dst = which == 0 ? p.dv : p.dk;
    const int wi = threadIdx.x >> 5, ln = threadIdx.x & 31;
#pragma unroll
    for (int j = 0; j < 128 / (16 * kRpi); ++j) {
      const int row = wi * (128 / 16) + j * kRpi + ln / kCpr;
      const int ch = ln % kCpr;
      const uint4 v = *reinterpret_cast<const uint4*>(stg + row * (2 * D) +
                                                      ((ch ^ (row & (kCpr - 1))) * 16));
      if (row >= f.kt.shift && row < f.kt.shift + f.kt.n) {
        const long long tok = f.off0 + f.kb * kBN - f.kt.shift + row;
        *reinterpret_cast<uint4*>(dst + (tok * p.Hkv + f.h) * D + ch * 8) = v;
      }
    }
    return true;
  };
  // dK of item itf, then its K buffer back to the producer (a TMA load may
  // follow the generic-proxy accesses above): every math thread arrives, and
  // once more the store warp after its store has read a full block, or
  // thread 0 for a ragged one.
  auto epi_dk = [&](const KvItem& f, uint32_t itf) {
    const bool full = f.kt.shift == 0 && f.kt.n == kBN;
    if (!epi_tensor(f, itf, 1, full)) return false;
    fence_proxy_async_smem();
    mbar_arrive(&c->k_empty[itf & 1]);
    if (!full && threadIdx.x == 0) mbar_arrive(&c->k_empty[itf & 1]);
    return true;
  };
  bool ok = true;
  uint32_t n = 0;
  KvItem f;
  uint32_t pk[16];
  // The math warps keep an item's slot of the item ring until its dK has
  // left TMEM.  The previous item's dK epilogue follows this item's first dS
  // part, so that the issuer's dK(g0) waits for one TMEM load rather than
  // for the whole epilogue; the previous item is read back from its slot.
  const bool any = next_item(c, n++, &f, &ok, p.err, false) && p_part(f, 0, gq, pk);
  // fin: a last pass that only runs the last item's dK epilogue (from the
  // same place in the loop as every other item's).
  bool fin = false;
  while (any) {
    bool fine = true;
    for (int i = 0; i < f.nt; ++i) {
      const uint32_t g = gq + i;
      if (!fin) {
        if (i > 0 && !p_part(f, i, g, pk)) { fine = false; break; }
        if (!ds_part(g, pk)) { fine = false; break; }
      }
      if (i == 0 && it > 0) {
        const uint32_t slot = (n - 2) & 1;
        if (!epi_dk(c->item[slot], it - 1)) { fine = false; break; }
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(&c->item_empty[slot]);
      }
      if (fin) break;
    }
    if (!fine || fin) break;
    // The next item's first P part comes before this item's epilogue: its
    // S^T is issued right after this item's last dK.
    KvItem fn;
    const bool have_n = next_item(c, n++, &fn, &ok, p.err, false);
    if (!ok) break;
    if (have_n && !p_part(fn, 0, gq + f.nt, pk)) break;
    if (!mbar_wait_warp(&c->dkdv_full, it & 1, &c->abort, p.err)) break;
    tc_fence_after();
    if (!epi_tensor(f, it, 0, f.kt.shift == 0 && f.kt.n == kBN)) break;
    gq += f.nt;
    ++it;
    if (have_n)
      f = fn;
    else
      fin = true;
  }
  // No more tensors for the store warp.
  if (threadIdx.x == 0) c->job[ns & 1].which = -1;
  mbar_arrive(&c->stg_full[ns & 1]);
}

// Store warp (one thread): TMA stores of the staged full blocks, in order.
// After dV's store has read the buffer, the math warps may stage dK there;
// after dK's, the K buffer goes back to the producer.
template <int D>
__device__ void store_role(const CUtensorMap* tdk, const CUtensorMap* tdv, uint8_t* smem,
                           KvCtl* c, int* err) {
  for (uint32_t e = 0;; ++e) {
    if (!mbar_wait(&c->stg_full[e & 1], (e >> 1) & 1, &c->abort, err)) break;
    const StoreJob j = c->job[e & 1];
    if (j.which < 0) break;
#pragma unroll
    for (int s = 0; s < D / 64; ++s)
      tma_store_3d(j.which == 0 ? tdv : tdk, smem + j.buf + s * 16384, s * 64, j.h, j.row);
    bulk_commit();
    bulk_wait_read0();
    mbar_arrive(j.which == 0 ? &c->stg_empty : &c->k_empty[j.kbuf]);
  }
  // The stores are complete before the CTA's shared memory goes away.
  bulk_wait0();
}

template <int D, bool LOCAL, bool BCAST, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kv_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                  const __grid_constant__ CUtensorMap tdk, const __grid_constant__ CUtensorMap tdv,
                  const __grid_constant__ CUtensorMap tq_h,
                  const __grid_constant__ CUtensorMap tdo_h, const BwdParams p) {
  using C = KvCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  KvCtl* c = reinterpret_cast<KvCtl*>(smem + C::kCtl);
  const int warp = warp_id(), lane = lane_id();
  const int rank = PAIR ? static_cast<int>(cluster_rank()) : 0;
  // Dynamic shared memory starts at the same offset in every CTA of the
  // kernel, so both CTAs of a pair take this exit together.
  if ((smem_addr(smem) & 1023) != 0) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrSmemAlign);
    return;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c->k_full[i], 1);
      // released by the math warps' epilogue and the store warp (a ragged
      // block: math thread 0 twice)
      mbar_init(&c->k_empty[i], kMath + 1);
    }
    mbar_init(&c->v_full, 1);
    mbar_init(&c->v_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c->q_full[i][0], 1);
      mbar_init(&c->q_full[i][1], 1);
      mbar_init(&c->q_empty[i], 1);
      mbar_init(&c->do_full[i][0], 1);
      mbar_init(&c->do_full[i][1], 1);
      mbar_init(&c->do_empty[i], 1);
      mbar_init(&c->stat_full[i], 1);
      mbar_init(&c->stat_empty[i], kMathWarps);  // after each math warp's dS part
      mbar_init(&c->item_full[i], 1);
      // math warps + the MMA warp (a pair's second CTA issues nothing)
      mbar_init(&c->item_empty[i], kMathWarps + (rank == 0 ? 1 : 0));
    }
    // Issued products: one commit arrives (on both CTAs of a pair).  Math
    // results for the issuer: every math thread, or one arrive per warp of
    // both CTAs of a pair.
    constexpr uint32_t kToIssuer = PAIR ? 2 * kMathWarps : kMath;
    mbar_init(&c->s_full, 1);
    mbar_init(&c->dp_full, 1);
    mbar_init(&c->p_full, kToIssuer);
    mbar_init(&c->ds_full, kToIssuer);
    mbar_init(&c->dkdv_full, 1);
    mbar_init(&c->dv_empty, kToIssuer);
    mbar_init(&c->dk_empty, kToIssuer);
    mbar_init(&c->epi, kMath);
    mbar_init(&c->stg_full[0], kMath);
    mbar_init(&c->stg_full[1], kMath);
    mbar_init(&c->stg_empty, 1);
    mbar_init(&c->drain, 1);
    c->abort = 0;
    fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    tma_prefetch_desc(&tdo);
    tma_prefetch_desc(&tdk);
    tma_prefetch_desc(&tdv);
    if (PAIR) {
      tma_prefetch_desc(&tq_h);
      tma_prefetch_desc(&tdo_h);
    }
  }
  if (warp == kMmaWarp) {  // a pair: one warp of each CTA, together
    if (PAIR) {
      tmem_alloc_pair(&c->tmem_base, 512);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&c->tmem_base, 512);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  // a pair: both CTAs' barriers exist before either signals the other's
  if (PAIR) cluster_sync();
  tc_fence_after();
  const uint32_t tbase = c->tmem_base;
  if (warp < kMathWarps) {
    math_role<D, LOCAL, BCAST, PAIR>(p, smem, c, tbase);
  } else if (warp == kStoreWarp) {
    if (lane == 0) store_role<D>(&tdk, &tdv, smem, c, p.err);
  } else if (warp == kProducerWarp) {
    if (lane == 0) producer_role<D, LOCAL, BCAST, PAIR>(&tq, &tk, &tv, &tdo, &tq_h, &tdo_h, p, smem, c);
  } else if (!PAIR || rank == 0) {
    mma_role<D, LOCAL, PAIR>(p, smem, c, tbase);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  // a pair: neither CTA leaves (or frees TMEM) while the other may still
  // signal its barriers or read its operands
  if (PAIR) cluster_sync();
  if (warp == kMmaWarp) {
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tbase, 512);
    else
      tmem_dealloc(tbase, 512);
  }
}

template <int D, bool LOCAL, bool BCAST, bool PAIR = false>
cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                     const CUtensorMap& tq_h, const CUtensorMap& tdo_h, const BwdParams& p,
                     int grid, cudaStream_t s) {
  using C = KvCfg<D>;
  static_assert(C::kSmem <= 232448, "shared memory budget");
  static_assert(sizeof(KvCtl) <= 512, "control block");
  static_assert(!(LOCAL && BCAST), "causal masking is self-attention only");
  static_assert(!PAIR || (D == 128 && !LOCAL), "pairs: D = 128 without a local mask");
  auto kern = bwd_kv_kernel<D, LOCAL, BCAST, PAIR>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  if (!PAIR) {
    kern<<<grid, kThreads, C::kSmem, s>>>(tq, tk, tv, tdo, tdk, tdv, tq_h, tdo_h, p);
    return cudaGetLastError();
  }
  // Clusters of two CTAs; as many pairs as can be resident at once (each
  // walks the list in a fixed stride, so fewer resident pairs only cost time).
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int pairs = grid / 2;
  cfg.gridDim = dim3(2 * pairs);
  int active = 0;
  if (cudaOccupancyMaxActiveClusters(&active, kern, &cfg) == cudaSuccess && active > 0)
    pairs = std::min(pairs, active);
  else
    (void)cudaGetLastError();
  pairs = std::max(pairs, 1);
  cfg.gridDim = dim3(2 * pairs);
  return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, tdo, tdk, tdv, tq_h, tdo_h, p);
}

}  // namespace

cudaError_t launch_bwd_kv(int D, bool causal, bool bcast, const CUtensorMap& tq,
                          const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                          const CUtensorMap& tdk, const CUtensorMap& tdv, const BwdParams& p,
                          int grid, cudaStream_t s, const CUtensorMap* tq_h,
                          const CUtensorMap* tdo_h) {
  if (bcast && causal) return cudaErrorInvalidValue;
  if (tq_h != nullptr || tdo_h != nullptr) {  // pairs of CTAs
    if (D != 128 || causal || tq_h == nullptr || tdo_h == nullptr) return cudaErrorInvalidValue;
    if (bcast)
      return launch_t<128, false, true, true>(tq, tk, tv, tdo, tdk, tdv, *tq_h, *tdo_h, p, grid, s);
    return launch_t<128, false, false, true>(tq, tk, tv, tdo, tdk, tdv, *tq_h, *tdo_h, p, grid, s);
  }
  if (D == 128) {
    if (bcast) return launch_t<128, false, true>(tq, tk, tv, tdo, tdk, tdv, tq, tdo, p, grid, s);
    if (causal) return launch_t<128, true, false>(tq, tk, tv, tdo, tdk, tdv, tq, tdo, p, grid, s);
    return launch_t<128, false, false>(tq, tk, tv, tdo, tdk, tdv, tq, tdo, p, grid, s);
  }
  if (bcast) return launch_t<64, false, true>(tq, tk, tv, tdo, tdk, tdv, tq, tdo, p, grid, s);
  if (causal) return launch_t<64, true, false>(tq, tk, tv, tdo, tdk, tdv, tq, tdo, p, grid, s);
  return launch_t<64, false, false>(tq, tk, tv, tdo, tdk, tdv, tq, tdo, p, grid, s);
}

}  // namespace jfa
