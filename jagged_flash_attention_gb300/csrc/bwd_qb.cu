// Broadcast-Q backward, pass 2 of 2: dQ for sm_103a.
//
// In broadcast-Q mode ("Optimizing Jagged Flash Attention with TLX",
// section 1, "The Challenge") every sequence attends with the same dense Q,
// so dQ of a query tile sums over the key tiles of ALL sequences:
//   dQ_t = scale * sum_b sum_j dS_{b,t,j} K_{b,j}.
// This pass cuts that sum into equal chunks of the concatenated key-tile
// stream; an item is (head, pair of 128-row query tiles, chunk).  dQ of both
// query tiles accumulates in tensor memory over the whole chunk, across
// sequence boundaries, and the item writes one fp32 partial; a finalize
// kernel sums the partials of each (head, pair) in a fixed order, so dQ is
// deterministic.  This stands in for the per-(key block, query tile)
// reduce-add across CTAs of the page's fused design (section 2.2,
// "Multi-stage dQ staging"): the reduction shrinks to one partial per item.
// Per query tile g and key tile u of the chunk (of sequence b):
//   S    = Q_g K_u^T        (SS)                -> TMEM SP_g
//   P    = exp2(S * scale*log2e - LSE_b*log2e)     (math, bf16 pairs in registers)
//   dP   = dO_{b,g} V_u^T   (SS)                -> TMEM SP_g (over S, once S is read)
//   dS   = P (dP - Delta_b): the difference in fp32, rounded to bf16, times
//          the bf16 P; packed into SP_g (keys 0-63 at +0, 64-127 at +64)
//   dQ_g += dS K_u          (TS, B = K MN-major) -> TMEM DQ_g
// Q is loaded once per item; dO and the row statistics once per sequence
// segment of the chunk.  dO has one barrier pair per query tile, so the next
// sequence's dO_g loads as soon as this sequence's last dP_g has read it.
// Issue order per key tile u: dQ_0(u-1) S_0(u) | dQ_1(u-1) S_1(u) | dP_0(u) |
// dP_1(u), as in the self-attention dQ pass, so each tile's score math runs
// under the other tile's products.
//
// CTA = 10 warps: warps 0-7 score math (warp w: TMEM lanes 32*(w%4).. =
// query rows of both tiles, key columns 64*(w/4)..) and the partial stores,
// warp 8 TMA producer, warp 9 MMA issuer.  TMEM (512 columns): tile g uses
// SP at 256g (128 fp32 columns) and DQ at 256g + 128 (D columns).
#include "common.cuh"
#include "ptx.cuh"

namespace jfa {
namespace {

constexpr int kThreads = 320;
constexpr int kMath = 256;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;

template <int D>
struct QbCfg {
  static constexpr int NSK = (D == 128) ? 2 : 3;   // K ring depth
  static constexpr int NSV = (D == 128) ? 1 : 3;   // V ring depth
  static constexpr int NSDO = (D == 128) ? 1 : 2;  // dO / statistics stages (sequence segments)
  static constexpr int kTile = kBM * D * 2;        // bytes of a 128-row bf16 tile
  static constexpr int kSlabs = D / 64;
  static constexpr int kStatBytes = 2 * kBM * 8;  // both query tiles of a segment
  static constexpr int kQ = 0;                     // query tile g at g * kTile
  static constexpr int kDO = 2 * kTile;            // stage s, tile g at kDO + (2s + g) * kTile
  static constexpr int kK = kDO + 2 * NSDO * kTile;
  static constexpr int kV = kK + NSK * kTile;
  static constexpr int kStat = kV + NSV * kTile;  // stage s at kStat + s * kStatBytes
  static constexpr int kCtl = kStat + NSDO * kStatBytes;
  static constexpr int kSmem = kCtl + 512;
};

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

// Item as decoded by the producer.  n < 0: no more items.
struct QbDec {
  int b, j, n;  // first sequence, its first key tile, key tiles of the chunk
  int h, pair, slot;
  int nt;  // query tiles of the pair (1 or 2)
};


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

struct QbCtl {
  uint64_t q_full, q_empty;
  uint64_t do_full[2][2], do_empty[2][2];  // [stage][query tile]
  uint64_t st_full[2], st_empty[2];        // [stage]
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], p_done[2], dp_full[2], ds_full[2];  // per query tile
  uint64_t dq_full[2], dq_free[2];
  uint64_t item_full[2], item_empty[2];
  uint64_t drain;
  QbDec item[2];
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, int* err) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > JFA_WAIT_LIMIT_CYCLES) {
      atomicOr(err, kErrTimeout);
      return;
    }
  }
}

__device__ __forceinline__ bool next_item(QbCtl* c, uint32_t n, QbDec* f, bool* ok, int* err) {
  const int slot = n & 1;
  if (!mbar_wait_warp(&c->item_full[slot], (n >> 1) & 1, &c->abort, err)) {
    *ok = false;
    return false;
  }
  *f = c->item[slot];
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&c->item_empty[slot]);
  return f->n >= 0;
}

template <int D>
__device__ void producer_role(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                              const CUtensorMap* tdo, const BwdParams& p, uint8_t* smem,
                              QbCtl* c) {
  using C = QbCfg<D>;
  const int n_items = p.hdr->n_items;
  const int T = p.hdr->T;
  const long long lq_pad = static_cast<long long>(cdiv(p.Lq, kBM)) * kBM;
  uint32_t itq = 0, nk = 0, nv = 0, gs = 0, gst = 0;  // gs / gst: dO / statistics segments
  bool ok = true;
  for (uint32_t n = 0; ok; ++n) {
    const int slot = n & 1;
    if (!mbar_wait(&c->item_empty[slot], ((n >> 1) & 1) ^ 1, &c->abort, p.err)) break;
    const int idx = atomicAdd(&p.hdr->ticket, 1);
    QbDec f;
    if (idx < n_items) {
      const QbItem it = p.qb_items[idx];
      f.h = it.hp & 0xffff;
      f.pair = it.hp >> 16;
      f.b = it.b;
      f.j = it.j;
      f.n = it.n;
      f.slot = idx;
      f.nt = min(2, cdiv(p.Lq - f.pair * kQbRows, kBM));
    } else {
      f.n = -1;
    }
    c->item[slot] = f;
    mbar_arrive(&c->item_full[slot]);
    if (idx >= n_items) break;
    if (f.n == 0) continue;
    if (!mbar_wait(&c->q_empty, (itq & 1) ^ 1, &c->abort, p.err)) break;
    mbar_arrive_expect_tx(&c->q_full, f.nt * C::kTile);
    for (int g = 0; g < f.nt; ++g)
#pragma unroll
      for (int s = 0; s < C::kSlabs; ++s)
        tma_load_3d(smem + C::kQ + g * C::kTile + s * 16384, tq, &c->q_full, s * 64, f.h,
                    f.pair * kQbRows + g * kBM);
    ++itq;
    Seg sg;
    seg_load(sg, p.offsets, p.B, f.b, f.j);
    for (int u = 0; u < f.n && ok; ++u) {
      const KvTile kt = kv_tile(sg.off0, sg.L, sg.j, T);
      {
        const int st = nk % C::NSK;
        if (!mbar_wait(&c->k_empty[st], ((nk / C::NSK) & 1) ^ 1, &c->abort, p.err)) { ok = false; break; }
        mbar_arrive_expect_tx(&c->k_full[st], C::kTile);
#pragma unroll
        for (int s = 0; s < C::kSlabs; ++s)
          tma_load_3d(smem + C::kK + st * C::kTile + s * 16384, tk, &c->k_full[st], s * 64,
                      f.h / p.G,
                      kt.row);
        ++nk;
      }
      if (u == 0 || sg.j == 0) {
        // A new sequence segment: its dO tiles and row statistics.  Both
        // tile barriers of the stage complete once per segment (a pair with
        // one query tile arrives on the second without a copy), so their
        // phases stay in step with the segment count.
        // The statistics first (their stage was read by the math at the
        // start of an earlier segment), then dO, whose stage frees only
        // after the previous segment's last dP.  Each load group counts
        // itself once issued, so the drain below sees every copy.  Both dO
        // tile barriers of a stage complete once per segment (a pair with
        // one query tile arrives on the second without a copy), so their
        // phases stay in step with the segment count.
        const int st = gs % C::NSDO;
        const uint32_t ph = ((gs / C::NSDO) & 1) ^ 1;
        if (!mbar_wait(&c->st_empty[st], ph, &c->abort, p.err)) { ok = false; break; }
        mbar_arrive_expect_tx(&c->st_full[st], f.nt * (C::kStatBytes / 2));
        const long long row0 = (static_cast<long long>(sg.b) * p.H + f.h) * lq_pad + f.pair * kQbRows;
        for (int g = 0; g < f.nt; ++g)
          bulk_load(smem + C::kStat + st * C::kStatBytes + g * (C::kStatBytes / 2),
                    p.stat + stat_float(row0 + g * kBM), C::kStatBytes / 2, &c->st_full[st]);
        ++gst;
        if (!mbar_wait(&c->do_empty[st][0], ph, &c->abort, p.err) ||
            !mbar_wait(&c->do_empty[st][1], ph, &c->abort, p.err)) {
          ok = false;
          break;
        }
        for (int g = 0; g < 2; ++g) {
          if (g < f.nt) {
            mbar_arrive_expect_tx(&c->do_full[st][g], C::kTile);
#pragma unroll
            for (int s = 0; s < C::kSlabs; ++s)
              tma_load_4d(smem + C::kDO + (2 * st + g) * C::kTile + s * 16384, tdo,
                          &c->do_full[st][g], s * 64, f.h, f.pair * kQbRows + g * kBM, sg.b);
          } else {
            mbar_arrive(&c->do_full[st][g]);
          }
        }
        ++gs;
      }
      {
        const int st = nv % C::NSV;
        if (!mbar_wait(&c->v_empty[st], ((nv / C::NSV) & 1) ^ 1, &c->abort, p.err)) { ok = false; break; }
        mbar_arrive_expect_tx(&c->v_full[st], C::kTile);
#pragma unroll
        for (int s = 0; s < C::kSlabs; ++s)
          tma_load_3d(smem + C::kV + st * C::kTile + s * 16384, tv, &c->v_full[st], s * 64,
                      f.h / p.G,
                      kt.row);
        ++nv;
      }
      if (u + 1 < f.n) seg_next(sg, p.offsets, p.B);
    }
  }
  // Drain: every copy this CTA issued has landed before exit.
  if (itq > 0) drain_wait(&c->q_full, (itq - 1) & 1, p.err);
  for (uint32_t g = nk > C::NSK ? nk - C::NSK : 0; g < nk; ++g)
    drain_wait(&c->k_full[g % C::NSK], (g / C::NSK) & 1, p.err);
  for (uint32_t g = nv > C::NSV ? nv - C::NSV : 0; g < nv; ++g)
    drain_wait(&c->v_full[g % C::NSV], (g / C::NSV) & 1, p.err);
  for (uint32_t g = gs > C::NSDO ? gs - C::NSDO : 0; g < gs; ++g) {
    drain_wait(&c->do_full[g % C::NSDO][0], (g / C::NSDO) & 1, p.err);
    drain_wait(&c->do_full[g % C::NSDO][1], (g / C::NSDO) & 1, p.err);
  }
  for (uint32_t g = gst > C::NSDO ? gst - C::NSDO : 0; g < gst; ++g)
    drain_wait(&c->st_full[g % C::NSDO], (g / C::NSDO) & 1, p.err);
}

template <int D>
__device__ void mma_role(const BwdParams& p, uint8_t* smem, QbCtl* c, uint32_t tbase) {
  using C = QbCfg<D>;
  const uint32_t leader = elect_one();
  const uint32_t id_s = idesc_bf16_f32(128, 128, false, false);  // S, dP
  const uint32_t id_dq = idesc_bf16_f32(128, D, false, true);    // dQ (A = dS in TMEM)
  const uint64_t dq_k0 = smem_desc_sw128(smem_addr(smem + C::kQ), 16, 1024);
  const uint64_t ddo_k0 = smem_desc_sw128(smem_addr(smem + C::kDO), 16, 1024);
  const uint64_t dk_k0 = smem_desc_sw128(smem_addr(smem + C::kK), 16, 1024);
  const uint64_t dk_m0 = smem_desc_sw128(smem_addr(smem + C::kK), 16384, 1024);
  const uint64_t dv_k0 = smem_desc_sw128(smem_addr(smem + C::kV), 16, 1024);
  auto issue_s = [&](int g, uint32_t kidx) {
    const uint64_t dq = desc_add(dq_k0, g * C::kTile);
    const uint64_t dk = desc_add(dk_k0, (kidx % C::NSK) * C::kTile);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
      if (leader) mma_ss(tbase + 256 * g, desc_add(dq, off), desc_add(dk, off), id_s, k > 0);
    }
  };
  auto issue_dp = [&](int g, uint32_t vidx, int st) {
    const uint64_t ddo = desc_add(ddo_k0, (2 * st + g) * C::kTile);
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
      if (leader)
        mma_ts(tbase + 256 * g + 128, tbase + 256 * g + 8 * k + (k >= 4 ? 32 : 0),
               desc_add(dk, k * 2048), id_dq, acc || (k > 0));
  };
  uint32_t itq = 0, nk = 0, nv = 0, gs = 0;
  uint32_t gt[2] = {0, 0};  // key tiles processed per query tile slot, over all items
  uint32_t gi[2] = {0, 0};  // items in which the slot was present
  bool ok = true, issued = false;
  for (uint32_t n = 0; ok; ++n) {
    QbDec f;
    if (!next_item(c, n, &f, &ok, p.err)) break;
    if (f.n == 0) continue;
    if (!mbar_wait_warp(&c->q_full, itq & 1, &c->abort, p.err)) break;
    ++itq;
    const int nt = f.nt;
    const uint32_t k0 = nk, v0 = nv;
    Seg sg;
    seg_load(sg, p.offsets, p.B, f.b, f.j);
    int st = 0;
    for (int u = 0; u <= f.n && ok; ++u) {
      bool k_ready = false;
      for (int g = 0; g < nt; ++g) {
        if (u >= 1) {
          if (!mbar_wait_warp(&c->ds_full[g], (gt[g] + u - 1) & 1, &c->abort, p.err)) { ok = false; break; }
          if (u == 1 && !mbar_wait_warp(&c->dq_free[g], (gi[g] & 1) ^ 1, &c->abort, p.err)) { ok = false; break; }
          tc_fence_after();
          issue_dq(g, k0 + u - 1, u > 1);
          if (u == f.n && leader) mma_commit(&c->dq_full[g]);
        }
        if (u < f.n) {
          if (!k_ready) {
            const uint32_t kk = k0 + u;
            if (!mbar_wait_warp(&c->k_full[kk % C::NSK], (kk / C::NSK) & 1, &c->abort, p.err)) { ok = false; break; }
            k_ready = true;
          }
          tc_fence_after();
          issue_s(g, k0 + u);
          if (leader) mma_commit(&c->s_full[g]);
          issued = true;
        }
      }
      if (!ok) break;
      if (u >= 1 && leader) mma_commit(&c->k_empty[(k0 + u - 1) % C::NSK]);  // K(u-1) fully read
      if (u < f.n) {
        const bool seg_start = u == 0 || sg.j == 0;
        const bool seg_end = u == f.n - 1 || sg.j == sg.nts - 1;
        if (seg_start) st = gs % C::NSDO;
        const uint32_t vv = v0 + u;
        if (!mbar_wait_warp(&c->v_full[vv % C::NSV], (vv / C::NSV) & 1, &c->abort, p.err)) { ok = false; break; }
        for (int g = 0; g < nt; ++g) {
          if (seg_start &&
              !mbar_wait_warp(&c->do_full[st][g], (gs / C::NSDO) & 1, &c->abort, p.err)) { ok = false; break; }
          if (!mbar_wait_warp(&c->p_done[g], (gt[g] + u) & 1, &c->abort, p.err)) { ok = false; break; }
          tc_fence_after();
          issue_dp(g, vv, st);
          if (leader) mma_commit(&c->dp_full[g]);
        }
        if (!ok) break;
        if (seg_end) {  // dO of the segment fully read (both tile barriers stay in step)
          if (leader) {
            mma_commit(&c->do_empty[st][0]);
            mma_commit(&c->do_empty[st][1]);
          }
          ++gs;
        }
        if (leader) mma_commit(&c->v_empty[vv % C::NSV]);
        if (u == f.n - 1 && leader) mma_commit(&c->q_empty);  // Q is read by S only
        if (u + 1 < f.n) seg_next(sg, p.offsets, p.B);
      }
    }
    if (!ok) break;
    for (int g = 0; g < nt; ++g) {
      gt[g] += f.n;
      gi[g] += 1;
    }
    nk += f.n;
    nv += f.n;
  }
  if (issued && leader) {
    mma_commit(&c->drain);
    drain_wait(&c->drain, 0, p.err);
  }
}

template <int D>
__device__ void math_role(const BwdParams& p, uint8_t* smem, QbCtl* c, uint32_t tbase) {
  using C = QbCfg<D>;
  const int r = threadIdx.x & 127;    // query row of each tile == TMEM lane
  const int half = threadIdx.x >> 7;  // key columns [64*half, 64*half + 64)
  const uint32_t lane_base = static_cast<uint32_t>((r >> 5) * 32) << 16;
  const int T = p.hdr->T;
  const float sl2 = p.scale_log2;
  const uint64_t sl2x2 = f2_pack(sl2, sl2);
  uint32_t gt[2] = {0, 0};
  uint32_t gi[2] = {0, 0};
  uint32_t gs = 0;
  bool ok = true;
  for (uint32_t n = 0; ok; ++n) {
    QbDec f;
    if (!next_item(c, n, &f, &ok, p.err)) break;
    if (f.n == 0) continue;
    const int nt = f.nt;
    // -LSE*log2e and -Delta of this row for the current segment's sequence
    // (padding rows past q_len: -inf and 0, so P = 0 there).
    uint64_t nlse2[2] = {0, 0}, ndlt2[2] = {0, 0};
    auto p_part = [&](int g, uint32_t u, const KvTile& kt, uint32_t (&pk)[32]) {
      if (!mbar_wait_warp(&c->s_full[g], u & 1, &c->abort, p.err)) return false;
      tc_fence_after();
      const uint32_t ts = tbase + lane_base + 256 * g + 64 * half;
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
      if (kt.nk < kBN || kt.shift > 0) {
        // Ragged key tile: keep columns [shift, shift + nk) (relative to this
        // thread's first column: [lo, lo + span)).
        const int lo = kt.shift - 64 * half;
        const uint32_t span = kt.nk > 0 ? static_cast<uint32_t>(kt.nk) : 0u;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint32_t keep = (static_cast<uint32_t>(2 * i - lo) < span ? 0x0000ffffu : 0u) |
                                (static_cast<uint32_t>(2 * i + 1 - lo) < span ? 0xffff0000u : 0u);
          pk[i] &= keep;
        }
      }
      return true;
    };
    auto ds_part = [&](int g, uint32_t u, const uint32_t (&pk)[32]) {
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
    Seg sg;
    seg_load(sg, p.offsets, p.B, f.b, f.j);
    for (int u = 0; u < f.n && ok; ++u) {
      if (u == 0 || sg.j == 0) {
        const int st = gs % C::NSDO;
        if (!mbar_wait_warp(&c->st_full[st], (gs / C::NSDO) & 1, &c->abort, p.err)) { ok = false; break; }
        const float* sb = reinterpret_cast<const float*>(smem + C::kStat + st * C::kStatBytes);
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          if (g < nt) {
            const float* e = sb + g * 2 * kBM + stat_float(r);
            nlse2[g] = f2_pack(e[0], e[0]);
            ndlt2[g] = f2_pack(e[4], e[4]);
          }
        }
        mbar_arrive(&c->st_empty[st]);
        ++gs;
      }
      const KvTile kt = kv_tile(sg.off0, sg.L, sg.j, T);
      uint32_t p0[32], p1[32];
      if (!p_part(0, gt[0] + u, kt, p0)) { ok = false; break; }
      if (nt > 1 && !p_part(1, gt[1] + u, kt, p1)) { ok = false; break; }
      if (!ds_part(0, gt[0] + u, p0)) { ok = false; break; }
      if (nt > 1 && !ds_part(1, gt[1] + u, p1)) { ok = false; break; }
      if (u + 1 < f.n) seg_next(sg, p.offsets, p.B);
    }
    if (!ok) break;
    // The item's fp32 dQ partials (unscaled), this thread's half of the head
    // dimension of row r: part[slot][g][r][:], rows of the dense Q only (the
    // finalize reads no others).
    for (int g = 0; g < nt; ++g) {
      if (!mbar_wait_warp(&c->dq_full[g], gi[g] & 1, &c->abort, p.err)) { ok = false; break; }
      tc_fence_after();
      float* dst = p.dq_part + ((static_cast<long long>(f.slot) * 2 + g) * kBM + r) * D;
      const bool row_ok = f.pair * kQbRows + g * kBM + r < p.Lq;
#pragma unroll
      for (int ch = 0; ch < D / 64; ++ch) {
        const int dbase = (D / 2) * half + 32 * ch;
        uint32_t v[32];
        tmem_ld32(tbase + lane_base + 256 * g + 128 + dbase, v);
        tmem_wait_ld();
        if (row_ok) {
#pragma unroll
          for (int q = 0; q < 4; ++q) st_global_v8(dst + dbase + 8 * q, v + 8 * q);
        }
      }
      tc_fence_before();
      mbar_arrive(&c->dq_free[g]);
      ++gi[g];
    }
    if (!ok) break;
    for (int g = 0; g < nt; ++g) gt[g] += f.n;
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_qb_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                  const BwdParams p) {
  using C = QbCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  QbCtl* c = reinterpret_cast<QbCtl*>(smem + C::kCtl);
  const int warp = warp_id(), lane = lane_id();
  if ((smem_addr(smem) & 1023) != 0) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrSmemAlign);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(&c->q_full, 1);
    mbar_init(&c->q_empty, 1);
    for (int s = 0; s < 2; ++s) {
      for (int g = 0; g < 2; ++g) {
        mbar_init(&c->do_full[s][g], 1);
        mbar_init(&c->do_empty[s][g], 1);
      }
      mbar_init(&c->st_full[s], 1);
      mbar_init(&c->st_empty[s], kMath);
    }
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
      mbar_init(&c->item_full[g], 1);
      mbar_init(&c->item_empty[g], 9);  // 8 math warps + the MMA warp
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
    math_role<D>(p, smem, c, tbase);
  } else if (warp == kProducerWarp) {
    if (lane == 0) producer_role<D>(&tq, &tk, &tv, &tdo, p, smem, c);
  } else {
    mma_role<D>(p, smem, c, tbase);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int D>
cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     const CUtensorMap& tdo, const BwdParams& p, int grid, cudaStream_t s) {
  using C = QbCfg<D>;
  static_assert(C::kSmem <= 232448, "shared memory budget");
  static_assert(sizeof(QbCtl) <= 512, "control block");
  static_assert(C::NSK <= 4 && C::NSV <= 4 && C::NSDO <= 2, "ring depth");
  static_assert(128 + D <= 256, "TMEM columns per query tile");
  auto kern = bwd_qb_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, C::kSmem, s>>>(tq, tk, tv, tdo, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_qb(int D, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& tdo, const BwdParams& p,
                          int grid, cudaStream_t s) {
  if (D == 128) return launch_t<128>(tq, tk, tv, tdo, p, grid, s);
  return launch_t<64>(tq, tk, tv, tdo, p, grid, s);
}

}  // namespace jfa
