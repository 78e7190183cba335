// Self-attention backward, pass 2 of 2: dQ for sm_103a.
//
// The dQ part of the five backward products ("Optimizing Jagged Flash
// Attention with TLX", "2-CTA collaborative MMA") computed query-outer like
// the forward, so that dQ of a query tile accumulates in tensor memory over
// all of its key tiles and is written once, in bf16, with no cross-CTA
// reduction (the fp32 reduce-add the page stages for broadcast-Q, section
// "Multi-stage dQ staging", has no counterpart here).  Per query tile and
// key tile j:
//   S_j  = Q K_j^T      (SS)                  -> TMEM SP
//   P    = exp2(S * scale*log2e - LSE*log2e)    (math, kept in registers as bf16)
//   dP_j = dO V_j^T     (SS)                  -> TMEM SP (over S, once P is read)
//   dS   = P (dP - Delta): dP - Delta in fp32, then a bf16 pair product,
//          packed into SP (keys 0-63 at +0, keys 64-127 at +64)
//   dQ  += dS K_j       (TS, B = K MN-major)  -> TMEM DQ
// Each item is a pair of 128-row query tiles of one (sequence, head) that
// share every K / V tile, which halves the K / V bytes each SM must take in
// per product (an SM ingests about 48 B per cycle from L2; one 128-row tile
// at full tensor rate would need about 42).  The MMA issuer interleaves the
// two tiles,
//   dQ_0(j-1) S_0(j) | dQ_1(j-1) S_1(j) | dP_0(j) | dP_1(j)
// and all eight math warps work on both tiles in that order (P_0, P_1,
// dS_0, dS_1), so each tile's score math runs under the other tile's
// products at the full warp count.
//
// TMEM (512 columns): tile g uses SP at 256g (128 fp32 columns) and DQ at
// 256g + 128 (D columns).  SMEM: Q and dO of both tiles, a K ring and a V
// ring (D = 128: 128 + 64 + 32 KB).
//
// CTA = 10 warps: warps 0-7 score math (warp w: TMEM lanes 32*(w%4).. =
// query rows of both tiles, key columns 64*(w/4)..) and the dQ epilogues,
// warp 8 TMA producer, warp 9 MMA issuer.
#include "common.cuh"
#include "ptx.cuh"

namespace jfa {
namespace {

constexpr int kThreads = 320;
constexpr int kMath = 256;  // score-math threads
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;

template <int D>
struct QCfg {
  static constexpr int NSK = (D == 128) ? 2 : 4;  // K ring depth
  static constexpr int NSV = (D == 128) ? 1 : 4;  // V ring depth
  static constexpr int kTile = kBM * D * 2;       // bytes of a 128-row bf16 tile
  static constexpr int kSlabs = D / 64;
  // Q of tile g at (2g) * kTile, dO of tile g at (2g + 1) * kTile.
  static constexpr int kK = 4 * kTile;
  static constexpr int kV = kK + NSK * kTile;
  static constexpr int kCtl = kV + NSV * kTile;
  static constexpr int kSmem = kCtl + 512;
};


__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

struct QTile {
  int q_lo;   // local index of the tile's first query row
  int nq;     // valid query rows (<= 0: tile absent)
  int shift;  // rows the box was moved back to stay inside [0, T)
  int row;    // TMA row coordinate
  int j0;     // first key tile this query tile visits
  int n;      // key tiles it visits, [j0, j0 + n) (0: absent)
};

struct QItem {
  int b, h, hk, off0, L;  // sequence, query head, K/V head
  int J0, N;  // key tiles of the item: [J0, J0 + N), the union of its two tiles' ranges
  QTile t[2];
};

struct QCtl {
  uint64_t qdo_full, qdo_empty;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], p_done[2], dp_full[2], ds_full[2];  // per query tile
  uint64_t dq_full[2], dq_free[2];
  uint64_t item_full[2], item_empty[2];
  uint64_t drain;
  QItem item[2];  // decoded by the producer; b < 0: no more items
  uint32_t tmem_base;
  int abort;
};

// LOCAL: a local mask (causal or a sliding window, bounds p.wl / p.wr): a
// query tile visits only the key tiles holding admissible keys of its rows.
template <bool LOCAL>
__device__ __forceinline__ QItem decode(const BwdParams& p, int idx, int T) {
  QItem f;
  const Item it = p.items[idx];
  f.b = it.x;
  f.h = it.y >> 16;
  f.hk = f.h / p.G;
  const int pair = it.y & 0xffff;
  f.off0 = p.offsets[f.b];
  f.L = p.offsets[f.b + 1] - f.off0;
  int lo = 1 << 30, hi = 0;
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    QTile& q = f.t[g];
    q.q_lo = (2 * pair + g) * kBM;
    q.nq = min(kBM, f.L - q.q_lo);
    const int start = f.off0 + q.q_lo;
    q.shift = max(0, start + kBM - T);
    q.row = start - q.shift;
    q.j0 = 0;
    q.n = 0;
    if (q.nq > 0) {
      if (LOCAL)
        key_tiles(q.q_lo, q.q_lo + q.nq - 1, f.L, p.wl, p.wr, &q.j0, &q.n);
      else
        q.n = cdiv(f.L, kBN);
      lo = min(lo, q.j0);
      hi = max(hi, q.j0 + q.n);
    }
  }
  f.J0 = hi > 0 ? lo : 0;
  f.N = hi > 0 ? hi - lo : 0;
  return f;
}

struct KvTile {
  int row, shift, nk;
};
__device__ __forceinline__ KvTile kv_tile(int off0, int L, int j, int T) {
  KvTile k;
  const int start = off0 + j * kBN;
  k.shift = max(0, start + kBN - T);
  k.row = start - k.shift;
  k.nk = min(kBN, L - j * kBN);
  return k;
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
// warps).  False when the list is done or a wait gave up (then *ok is false).
__device__ __forceinline__ bool next_item(QCtl* c, uint32_t n, QItem* f, bool* ok, int* err) {
  const int slot = n & 1;
  if (!mbar_wait_warp(&c->item_full[slot], (n >> 1) & 1, &c->abort, err)) {
    *ok = false;
    return false;
  }
  *f = c->item[slot];
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&c->item_empty[slot]);
  return f->b >= 0;
}

template <int D, bool LOCAL>
__device__ void producer_role(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                              const CUtensorMap* tdo, const BwdParams& p, uint8_t* smem,
                              QCtl* c) {
  using C = QCfg<D>;
  const int n_items = p.hdr->n_items;
  const int T = p.hdr->T;
  uint32_t it = 0, nk = 0, nv = 0;
  bool ok = true;
  // One-item lookahead: the next item is taken and decoded while this one's
  // loads go out, and its Q / dO boxes and first K / V boxes are prefetched
  // into L2, so that at the item boundary they come from L2 rather than HBM.
  auto fetch = [&](QItem& f) {
    const int idx = atomicAdd(&p.hdr->ticket, 1);
    if (idx < n_items)
      f = decode<LOCAL>(p, idx, T);
    else
      f.b = -1;
  };
  auto prefetch = [&](const QItem& f) {
    const KvTile kt = kv_tile(f.off0, f.L, f.J0, T);
#pragma unroll
    for (int s = 0; s < C::kSlabs; ++s) {
#pragma unroll
      for (int g = 0; g < 2; ++g)
        if (f.t[g].n > 0 && f.t[g].row >= 0) {
          tma_prefetch_l2_3d(tq, s * 64, f.h, f.t[g].row);
          tma_prefetch_l2_3d(tdo, s * 64, f.h, f.t[g].row);
        }
      if (kt.row >= 0) {
        tma_prefetch_l2_3d(tk, s * 64, f.hk, kt.row);
        tma_prefetch_l2_3d(tv, s * 64, f.hk, kt.row);
      }
    }
  };
  QItem f, nx;
  fetch(f);
  for (uint32_t n = 0; ok; ++n, f = nx) {
    const int slot = n & 1;
    if (!mbar_wait(&c->item_empty[slot], ((n >> 1) & 1) ^ 1, &c->abort, p.err)) break;
    c->item[slot] = f;
    mbar_arrive(&c->item_full[slot]);
    if (f.b < 0) break;
    if (!mbar_wait(&c->qdo_empty, (it & 1) ^ 1, &c->abort, p.err)) break;
    const int ntiles = f.t[1].n > 0 ? 2 : 1;
    mbar_arrive_expect_tx(&c->qdo_full, ntiles * 2 * C::kTile);
    for (int g = 0; g < ntiles; ++g) {
#pragma unroll
      for (int s = 0; s < C::kSlabs; ++s) {
        tma_load_3d(smem + (2 * g) * C::kTile + s * 16384, tq, &c->qdo_full, s * 64, f.h,
                    f.t[g].row);
        tma_load_3d(smem + (2 * g + 1) * C::kTile + s * 16384, tdo, &c->qdo_full, s * 64, f.h,
                    f.t[g].row);
      }
    }
    ++it;
    for (int j = 0; j < f.N; ++j) {
      const KvTile kt = kv_tile(f.off0, f.L, (LOCAL ? f.J0 : 0) + j, T);
      {
        const int st = nk % C::NSK;
        if (!mbar_wait(&c->k_empty[st], ((nk / C::NSK) & 1) ^ 1, &c->abort, p.err)) { ok = false; break; }
        mbar_arrive_expect_tx(&c->k_full[st], C::kTile);
#pragma unroll
        for (int s = 0; s < C::kSlabs; ++s)
          tma_load_3d(smem + C::kK + st * C::kTile + s * 16384, tk, &c->k_full[st], s * 64, f.hk,
                      kt.row);
        ++nk;
      }
      {
        const int st = nv % C::NSV;
        if (!mbar_wait(&c->v_empty[st], ((nv / C::NSV) & 1) ^ 1, &c->abort, p.err)) { ok = false; break; }
        mbar_arrive_expect_tx(&c->v_full[st], C::kTile);
#pragma unroll
        for (int s = 0; s < C::kSlabs; ++s)
          tma_load_3d(smem + C::kV + st * C::kTile + s * 16384, tv, &c->v_full[st], s * 64, f.hk,
                      kt.row);
        ++nv;
      }
      if (j == 0) {  // after the item's first K / V loads
        fetch(nx);
        if (nx.b >= 0) prefetch(nx);
      }
    }
  }
  if (it > 0) drain_wait(&c->qdo_full, (it - 1) & 1, p.err);
  for (uint32_t g = nk > C::NSK ? nk - C::NSK : 0; g < nk; ++g)
    drain_wait(&c->k_full[g % C::NSK], (g / C::NSK) & 1, p.err);
  for (uint32_t g = nv > C::NSV ? nv - C::NSV : 0; g < nv; ++g)
    drain_wait(&c->v_full[g % C::NSV], (g / C::NSV) & 1, p.err);
}

template <int D, bool LOCAL>
__device__ void mma_role(const BwdParams& p, uint8_t* smem, QCtl* c, uint32_t tbase) {
  using C = QCfg<D>;
  // Run by the whole warp; the elected lane issues products and commits.
  const uint32_t leader = elect_one();
  const uint32_t id_s = idesc_bf16_f32(128, 128, false, false);  // S, dP
  const uint32_t id_dq = idesc_bf16_f32(128, D, false, true);    // dQ (A = dS in TMEM)
  // Descriptors built once; per tile and K step only adds remain.
  const uint64_t dq_k0 = smem_desc_sw128(smem_addr(smem), 16, 1024);
  const uint64_t dk_k0 = smem_desc_sw128(smem_addr(smem + C::kK), 16, 1024);
  const uint64_t dk_m0 = smem_desc_sw128(smem_addr(smem + C::kK), 16384, 1024);
  const uint64_t dv_k0 = smem_desc_sw128(smem_addr(smem + C::kV), 16, 1024);
  auto issue_s = [&](int g, uint32_t kidx) {
    const uint64_t dq = desc_add(dq_k0, (2 * g) * C::kTile);
    const uint64_t dk = desc_add(dk_k0, (kidx % C::NSK) * C::kTile);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
      if (leader) mma_ss(tbase + 256 * g, desc_add(dq, off), desc_add(dk, off), id_s, k > 0);
    }
  };
  auto issue_dp = [&](int g, uint32_t vidx) {
    const uint64_t ddo = desc_add(dq_k0, (2 * g + 1) * C::kTile);
    const uint64_t dv = desc_add(dv_k0, (vidx % C::NSV) * C::kTile);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
      if (leader) mma_ss(tbase + 256 * g, desc_add(ddo, off), desc_add(dv, off), id_s, k > 0);
    }
  };
  auto issue_dq = [&](int g, uint32_t kidx, bool acc) {
    // A = dS: bf16 pairs of keys 0-63 packed at SP + 0, of keys 64-127 at SP + 64.
    const uint64_t dk = desc_add(dk_m0, (kidx % C::NSK) * C::kTile);
#pragma unroll
    for (int k = 0; k < kBN / 16; ++k)
      if (leader) mma_ts(tbase + 256 * g + 128, tbase + 256 * g + 8 * k + (k >= 4 ? 32 : 0),
             desc_add(dk, k * 2048), id_dq, acc || (k > 0));
  };
  uint32_t it = 0, nk = 0, nv = 0;
  uint32_t gt[2] = {0, 0};  // tiles processed per query tile slot, over all items
  uint32_t gi[2] = {0, 0};  // items in which the slot was present
  bool ok = true, issued = false;
  for (uint32_t n = 0; ok; ++n) {
    QItem f;
    if (!next_item(c, n, &f, &ok, p.err)) break;
    if (!mbar_wait_warp(&c->qdo_full, it & 1, &c->abort, p.err)) break;
    const int N = f.N;
    const int nt[2] = {f.t[0].n, f.t[1].n};
    // step j of the item is key tile J0 + j; for query tile g it is its own
    // key tile lj = j + d[g] (active for 0 <= lj < nt[g])
    const int d[2] = {LOCAL ? f.J0 - f.t[0].j0 : 0, LOCAL ? f.J0 - f.t[1].j0 : 0};
    const uint32_t k0 = nk, v0 = nv;
    // Step j: dQ_g(j-1) and S_g(j) for both tiles, then dP_0(j), dP_1(j).
    for (int j = 0; j <= N && ok; ++j) {
      bool k_ready = false;
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const int lj = j + d[g];
        if (lj >= 1 && lj - 1 < nt[g]) {
          const uint32_t u = gt[g] + lj - 1;
          if (!mbar_wait_warp(&c->ds_full[g], u & 1, &c->abort, p.err)) { ok = false; break; }
          if (lj == 1 && !mbar_wait_warp(&c->dq_free[g], (gi[g] & 1) ^ 1, &c->abort, p.err)) { ok = false; break; }
          tc_fence_after();
          issue_dq(g, k0 + j - 1, lj > 1);
          if (lj == nt[g]) if (leader) mma_commit(&c->dq_full[g]);
        }
        if (lj >= 0 && lj < nt[g]) {
          if (!k_ready) {
            const uint32_t kk = k0 + j;
            if (!mbar_wait_warp(&c->k_full[kk % C::NSK], (kk / C::NSK) & 1, &c->abort, p.err)) { ok = false; break; }
            k_ready = true;
          }
          tc_fence_after();
          issue_s(g, k0 + j);
          if (leader) mma_commit(&c->s_full[g]);
          issued = true;
        }
      }
      if (!ok) break;
      if (j >= 1) if (leader) mma_commit(&c->k_empty[(k0 + j - 1) % C::NSK]);  // K(j-1) fully read
      if (j < N) {
        const uint32_t vv = v0 + j;
        if (!mbar_wait_warp(&c->v_full[vv % C::NSV], (vv / C::NSV) & 1, &c->abort, p.err)) { ok = false; break; }
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          const int lj = j + d[g];
          if (lj >= 0 && lj < nt[g]) {
            if (!mbar_wait_warp(&c->p_done[g], (gt[g] + lj) & 1, &c->abort, p.err)) { ok = false; break; }
            tc_fence_after();
            issue_dp(g, vv);
            if (leader) mma_commit(&c->dp_full[g]);
          }
        }
        if (!ok) break;
        if (leader) mma_commit(&c->v_empty[vv % C::NSV]);
        if (j == N - 1) if (leader) mma_commit(&c->qdo_empty);  // Q and dO are read by S and dP only
      }
    }
    if (!ok) break;
    gt[0] += nt[0];
    gt[1] += nt[1];
    gi[0] += nt[0] > 0 ? 1 : 0;
    gi[1] += nt[1] > 0 ? 1 : 0;
    nk += N;
    nv += N;
    ++it;
  }
  if (issued && leader) {
    mma_commit(&c->drain);
    drain_wait(&c->drain, 0, p.err);
  }
}

template <int D, bool LOCAL>
__device__ void math_role(const BwdParams& p, QCtl* c, uint32_t tbase) {
  const int r = threadIdx.x & 127;    // query row of each tile == TMEM lane
  const int half = threadIdx.x >> 7;  // key columns [64*half, 64*half + 64)
  const uint32_t lane_base = static_cast<uint32_t>((r >> 5) * 32) << 16;
  const int T = p.hdr->T;
  const float sl2 = p.scale_log2;
  const uint64_t sl2x2 = f2_pack(sl2, sl2);
  uint32_t gt[2] = {0, 0};  // tiles processed per query tile slot
  uint32_t gi[2] = {0, 0};  // items in which the slot was present
  bool ok = true;
  for (uint32_t n = 0; ok; ++n) {
    QItem f;
    if (!next_item(c, n, &f, &ok, p.err)) break;
    // Per query tile g of the item: this row's local query index, validity,
    // LSE*log2e and Delta.
    int qi[2];
    bool row_valid[2];
    uint64_t nlse2[2], ndlt2[2];
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      const QTile& q = f.t[g];
      qi[g] = q.q_lo - q.shift + r;
      row_valid[g] = q.n > 0 && r >= q.shift && r < q.shift + q.nq;
      float nl = -INFINITY, nd = 0.f;  // rows outside the sequence: P = 0
      if (row_valid[g]) {
        const long long si = static_cast<long long>(f.h) * T + f.off0 + qi[g];
        const float* st = p.stat + stat_float(stat_pos(si, 0));
        nl = st[0];  // -LSE*log2e
        nd = st[4];  // -Delta
      }
      nlse2[g] = f2_pack(nl, nl);
      ndlt2[g] = f2_pack(nd, nd);
    }
    // P of tile g at its key tile j (key tile t[g].j0 + j of the sequence):
    // this thread's 64 columns -> 32 bf16 pairs.
    auto p_part = [&](int g, int j, uint32_t (&pk)[32]) {
      const uint32_t u = gt[g] + j;
      if (!mbar_wait_warp(&c->s_full[g], u & 1, &c->abort, p.err)) return false;
      tc_fence_after();
      const uint32_t ts = tbase + lane_base + 256 * g + 64 * half;
      // All 64 columns leave TMEM first, so that dP may overwrite SP while
      // the exponentials are computed.
      uint32_t sraw[2][32];
      tmem_ld32(ts, sraw[0]);
      tmem_ld32(ts + 32, sraw[1]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&c->p_done[g]);  // S read: dP may overwrite SP
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 x = f2_unpack(ffma2(f2_pack(__uint_as_float(sraw[ch][2 * i]),
                                                   __uint_as_float(sraw[ch][2 * i + 1])),
                                           sl2x2, nlse2[g]));
          pk[16 * ch + i] = pack_bf16x2(ex2_approx(x.x), ex2_approx(x.y));
        }
      }
      const QTile& q = f.t[g];
      const int jk = LOCAL ? q.j0 + j : j;
      const KvTile kt = kv_tile(f.off0, f.L, jk, T);
      const int key0 = jk * kBN - kt.shift;  // local key index of column 0
      const int qa = q.q_lo - q.shift;       // local query index of row 0 of the box
      if (kt.nk < kBN || kt.shift > 0 ||
          (LOCAL && (key0 + kBN - 1 > qa + p.wr || key0 < qa + kBM - 1 - p.wl))) {
        // Ragged tile, or one that a band edge crosses: zero the
        // inadmissible columns.  The admissible ones are [lo, lo + span]
        // (relative to this thread's first column); an empty range moves lo
        // past every column.
        int first = kt.shift, last = kt.shift + kt.nk - 1;
        if (LOCAL) {  // admissible keys [qi - wl, qi + wr]
          first = max(first, qi[g] - p.wl - key0);
          last = min(last, qi[g] + p.wr - key0);
        }
        const int lo = (last >= first ? first : kBN) - 64 * half;
        const uint32_t span = last >= first ? static_cast<uint32_t>(last - first) : 0u;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint32_t keep = (static_cast<uint32_t>(2 * i - lo) <= span ? 0x0000ffffu : 0u) |
                                (static_cast<uint32_t>(2 * i + 1 - lo) <= span ? 0xffff0000u : 0u);
          pk[i] &= keep;
        }
      }
      return true;
    };
    // dS = P (dP - Delta) of tile g at key tile j, bf16 pairs into SP's
    // columns 64*half + [0, 32): inside this thread's own, already read
    // columns.
    auto ds_part = [&](int g, int j, const uint32_t (&pk)[32]) {
      const uint32_t u = gt[g] + j;
      if (!mbar_wait_warp(&c->dp_full[g], u & 1, &c->abort, p.err)) return false;
      tc_fence_after();
      const uint32_t ts = tbase + lane_base + 256 * g + 64 * half;
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t praw[32];
        tmem_ld32(ts + 32 * ch, praw);
        tmem_wait_ld();
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          // (dP - Delta) in fp32, rounded to bf16, times the bf16 P.
          const float2 d = f2_unpack(fadd2(
              f2_pack(__uint_as_float(praw[2 * i]), __uint_as_float(praw[2 * i + 1])), ndlt2[g]));
          w[i] = bmul2(pk[16 * ch + i], pack_bf16x2(d.x, d.y));
        }
        tmem_st16(ts + 16 * ch, w);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&c->ds_full[g]);
      return true;
    };
    // Per key tile j: P of both tiles, then dS of both tiles (in the order
    // the MMA issuer produces S_0, S_1, dP_0, dP_1).
    const int n0 = f.t[0].n, n1 = f.t[1].n;
    const int d0 = LOCAL ? f.J0 - f.t[0].j0 : 0, d1 = LOCAL ? f.J0 - f.t[1].j0 : 0;
    for (int j = 0; j < f.N && ok; ++j) {
      uint32_t p0[32], p1[32];
      const int l0 = j + d0, l1 = j + d1;  // the step in each tile's own key tiles
      const bool a0 = l0 >= 0 && l0 < n0, a1 = l1 >= 0 && l1 < n1;
      if (a0 && !p_part(0, l0, p0)) { ok = false; break; }
      if (a1 && !p_part(1, l1, p1)) { ok = false; break; }
      if (a0 && !ds_part(0, l0, p0)) { ok = false; break; }
      if (a1 && !ds_part(1, l1, p1)) { ok = false; break; }
    }
    if (!ok) break;
    // Epilogues: dQ = scale * acc in bf16 (this thread's half of the head dim).
#pragma unroll
    for (int g = 0; g < 2; ++g) {
      if (f.t[g].n == 0) continue;
      if (!mbar_wait_warp(&c->dq_full[g], gi[g] & 1, &c->abort, p.err)) { ok = false; break; }
      tc_fence_after();
      __nv_bfloat16* dst = p.dq + ((static_cast<long long>(f.off0) + qi[g]) * p.H + f.h) * D;
#pragma unroll
      for (int ch = 0; ch < D / 64; ++ch) {
        const int dbase = (D / 2) * half + 32 * ch;
        uint32_t v[32];
        tmem_ld32(tbase + lane_base + 256 * g + 128 + dbase, v);
        tmem_wait_ld();
        uint32_t w[16];
#pragma unroll
        for (int i2 = 0; i2 < 16; ++i2)
          w[i2] = pack_bf16x2(__uint_as_float(v[2 * i2]) * p.scale,
                              __uint_as_float(v[2 * i2 + 1]) * p.scale);
        if (row_valid[g]) st_global_64B(dst + dbase, w);
      }
      tc_fence_before();
      mbar_arrive(&c->dq_free[g]);
      ++gi[g];
    }
    gt[0] += n0;
    gt[1] += n1;
  }
}

template <int D, bool LOCAL>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_q_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                 const BwdParams p) {
  using C = QCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  QCtl* c = reinterpret_cast<QCtl*>(smem + C::kCtl);
  const int warp = warp_id(), lane = lane_id();
  if ((smem_addr(smem) & 1023) != 0) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrSmemAlign);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(&c->qdo_full, 1);
    mbar_init(&c->qdo_empty, 1);
    for (int i = 0; i < C::NSK; ++i) {
      mbar_init(&c->k_full[i], 1);
      mbar_init(&c->k_empty[i], 1);
    }
    for (int i = 0; i < C::NSV; ++i) {
      mbar_init(&c->v_full[i], 1);
      mbar_init(&c->v_empty[i], 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(&c->s_full[g], 1);
      mbar_init(&c->p_done[g], kMath);
      mbar_init(&c->dp_full[g], 1);
      mbar_init(&c->ds_full[g], kMath);
      mbar_init(&c->dq_full[g], 1);
      mbar_init(&c->dq_free[g], kMath);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c->item_full[i], 1);
      mbar_init(&c->item_empty[i], 9);  // 8 math warps + the MMA warp
    }
    mbar_init(&c->drain, 1);
    c->abort = 0;
    fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
    tma_prefetch_desc(&tdo);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&c->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = c->tmem_base;
  if (warp < 8) {
    math_role<D, LOCAL>(p, c, tbase);
  } else if (warp == kProducerWarp) {
    if (lane == 0) producer_role<D, LOCAL>(&tq, &tk, &tv, &tdo, p, smem, c);
  } else {
    mma_role<D, LOCAL>(p, smem, c, tbase);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int D, bool LOCAL>
cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     const CUtensorMap& tdo, const BwdParams& p, int grid, cudaStream_t s) {
  using C = QCfg<D>;
  static_assert(C::kSmem <= 232448, "shared memory budget");
  static_assert(sizeof(QCtl) <= 512, "control block");
  static_assert(C::NSK <= 4 && C::NSV <= 4, "ring depth");
  static_assert(128 + D <= 256, "TMEM columns per query tile");
  auto kern = bwd_q_kernel<D, LOCAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, C::kSmem, s>>>(tq, tk, tv, tdo, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_q(int D, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, const CUtensorMap& tdo, const BwdParams& p,
                         int grid, cudaStream_t s) {
  if (D == 128) {
    if (causal) return launch_t<128, true>(tq, tk, tv, tdo, p, grid, s);
    return launch_t<128, false>(tq, tk, tv, tdo, p, grid, s);
  }
  if (causal) return launch_t<64, true>(tq, tk, tv, tdo, p, grid, s);
  return launch_t<64, false>(tq, tk, tv, tdo, p, grid, s);
}

}  // namespace jfa
