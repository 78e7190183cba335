// Broadcast-Q backward with a short dense Q (q_len <= 128, D = 64), one pass
// for sm_103a.
//
// When the dense Q is one 128-row tile, all queries that attend to a key
// tile are in the CTA that processes it, so dV and dK of that key tile are
// complete after its products and need no accumulation across CTAs; dQ
// sums over every key tile of every sequence ("Optimizing Jagged Flash
// Attention with TLX", section 1, broadcast_q).  An item is a chunk of the
// key-tile stream of all sequences (as in the dQ pass of bwd_qb.cu): the CTA
// keeps Q, streams K and V, and per key tile u (of sequence b) computes the
// five products of the backward ("2-CTA collaborative MMA (backward)": S,
// dP, dV, dK, dQ) query-outer:
//   S    = Q K_u^T        (SS)                 -> TMEM SP
//   P    = exp2(S * scale*log2e - LSE_b*log2e)    (math; bf16, also written to
//          shared memory as P^T in the MN-major operand layout)
//   dP   = dO_b V_u^T     (SS)                 -> TMEM SP (over S)
//   dS   = P (dP - Delta_b): bf16 pairs packed into SP, and dS^T into shared
//          memory like P^T
//   dV_u = P^T dO_b       (SS, A = P^T MN-major, B = dO MN-major) -> TMEM dV[u&1]
//   dK_u = dS^T Q         (SS, A = dS^T MN-major, B = Q MN-major)  -> TMEM dK[u&1]
//   dQ  += dS K_u         (TS, A = dS in TMEM, B = K MN-major)     -> TMEM DQ
// dV_u, scale * dK_u are stored by the math warps while the next key tile
// runs (dV / dK double-buffered in TMEM); dQ leaves once per item as an fp32
// partial that the finalize kernel sums.  K and V are read once, so the
// pass moves the algorithmic bytes of the whole backward.  The products over
// queries (dV, dK) take only ceil(q_len / 16) K steps.
// Issue order per key tile u: dQ(u-1), dK(u-1) | S(u) | dP(u) | dV(u).
//
// CTA = 10 warps: warps 0-7 math (thread: TMEM lane = query row r, key
// columns 64 * half..; in the dV / dK epilogue, lane = key row, half 0 dV,
// half 1 dK), warp 8 TMA producer, warp 9 MMA issuer.  TMEM: SP [0,128),
// DQ [128,192), dV0 [192,256), dK0 [256,320), dV1 [320,384), dK1 [384,448).
#include "common.cuh"
#include "ptx.cuh"

namespace jfa {
namespace {

constexpr int D = 64;
constexpr int kThreads = 320;
constexpr int kMath = 256;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int NSK = 3, NSV = 3, NSDO = 2;
constexpr int kTile = kBM * D * 2;          // 16 KB: a 128-row bf16 tile (one 64-column slab)
constexpr int kStatBytes = kBM * 8;         // one query tile's statistics
constexpr int kQ = 0;
constexpr int kDO = kQ + kTile;             // stage s at kDO + s * kTile
constexpr int kK = kDO + NSDO * kTile;
constexpr int kV = kK + NSK * kTile;
constexpr int kPT = kV + NSV * kTile;       // P^T operand: 2 key chunks x 128 query rows x 128 B
constexpr int kDST = kPT + 2 * kTile;       // dS^T operand, same layout
constexpr int kStat = kDST + 2 * kTile;     // stage s at kStat + s * kStatBytes
constexpr int kCtl = kStat + NSDO * kStatBytes;
constexpr int kSmem = kCtl + 512;
constexpr uint32_t kColSP = 0, kColDQ = 128;
__host__ __device__ constexpr uint32_t col_dv(int buf) { return 192 + 128 * buf; }
__host__ __device__ constexpr uint32_t col_dk(int buf) { return 256 + 128 * buf; }

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

struct BsDec {
  int b, j, n, h, slot;
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

struct BsCtl {
  uint64_t q_full, q_empty;
  uint64_t do_full[NSDO], do_empty[NSDO], st_full[NSDO], st_empty[NSDO];
  uint64_t k_full[NSK], k_empty[NSK], v_full[NSV], v_empty[NSV];
  uint64_t s_full, p_done, p_full, dp_full, ds_full;
  uint64_t dkdv_full[2], dkdv_empty[2];
  uint64_t dq_full, dq_free;
  uint64_t item_full[2], item_empty[2];
  uint64_t drain;
  BsDec item[2];
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

__device__ __forceinline__ bool next_item(BsCtl* c, uint32_t n, BsDec* f, bool* ok, int* err) {
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

__device__ void producer_role(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                              const CUtensorMap* tdo, const BwdParams& p, uint8_t* smem,
                              BsCtl* c) {
  const int n_items = p.hdr->n_items;
  const int T = p.hdr->T;
  uint32_t itq = 0, nk = 0, nv = 0, gs = 0, gst = 0;
  bool ok = true;
  for (uint32_t n = 0; ok; ++n) {
    const int slot = n & 1;
    if (!mbar_wait(&c->item_empty[slot], ((n >> 1) & 1) ^ 1, &c->abort, p.err)) break;
    const int idx = atomicAdd(&p.hdr->ticket, 1);
    BsDec f;
    if (idx < n_items) {
      const QbItem it = p.qb_items[idx];
      f.h = it.hp & 0xffff;
      f.b = it.b;
      f.j = it.j;
      f.n = it.n;
      f.slot = idx;
    } else {
      f.n = -1;
    }
    c->item[slot] = f;
    mbar_arrive(&c->item_full[slot]);
    if (idx >= n_items) break;
    if (f.n == 0) continue;
    if (!mbar_wait(&c->q_empty, (itq & 1) ^ 1, &c->abort, p.err)) break;
    mbar_arrive_expect_tx(&c->q_full, kTile);
    tma_load_3d(smem + kQ, tq, &c->q_full, 0, f.h, 0);
    ++itq;
    Seg sg;
    seg_load(sg, p.offsets, p.B, f.b, f.j);
    for (int u = 0; u < f.n && ok; ++u) {
      const KvTile kt = kv_tile(sg.off0, sg.L, sg.j, T);
      {
        const int st = nk % NSK;
        if (!mbar_wait(&c->k_empty[st], ((nk / NSK) & 1) ^ 1, &c->abort, p.err)) { ok = false; break; }
        mbar_arrive_expect_tx(&c->k_full[st], kTile);
        tma_load_3d(smem + kK + st * kTile, tk, &c->k_full[st], 0, f.h, kt.row);
        ++nk;
      }
      if (u == 0 || sg.j == 0) {
        // A new sequence segment: statistics (their stage was read at the
        // start of an earlier segment), then dO (its stage frees after the
        // earlier segment's last dV).  Each group counts itself once issued.
        const int st = gs % NSDO;
        const uint32_t ph = ((gs / NSDO) & 1) ^ 1;
        if (!mbar_wait(&c->st_empty[st], ph, &c->abort, p.err)) { ok = false; break; }
        mbar_arrive_expect_tx(&c->st_full[st], kStatBytes);
        const long long lq_pad = kBM;  // q_len <= 128: one padded tile per sequence
        bulk_load(smem + kStat + st * kStatBytes,
                  p.stat + stat_float((static_cast<long long>(sg.b) * p.H + f.h) * lq_pad),
                  kStatBytes, &c->st_full[st]);
        ++gst;
        if (!mbar_wait(&c->do_empty[st], ph, &c->abort, p.err)) { ok = false; break; }
        mbar_arrive_expect_tx(&c->do_full[st], kTile);
        tma_load_4d(smem + kDO + st * kTile, tdo, &c->do_full[st], 0, f.h, 0, sg.b);
        ++gs;
      }
      {
        const int st = nv % NSV;
        if (!mbar_wait(&c->v_empty[st], ((nv / NSV) & 1) ^ 1, &c->abort, p.err)) { ok = false; break; }
        mbar_arrive_expect_tx(&c->v_full[st], kTile);
        tma_load_3d(smem + kV + st * kTile, tv, &c->v_full[st], 0, f.h, kt.row);
        ++nv;
      }
      if (u + 1 < f.n) seg_next(sg, p.offsets, p.B);
    }
  }
  if (itq > 0) drain_wait(&c->q_full, (itq - 1) & 1, p.err);
  for (uint32_t g = nk > NSK ? nk - NSK : 0; g < nk; ++g)
    drain_wait(&c->k_full[g % NSK], (g / NSK) & 1, p.err);
  for (uint32_t g = nv > NSV ? nv - NSV : 0; g < nv; ++g)
    drain_wait(&c->v_full[g % NSV], (g / NSV) & 1, p.err);
  for (uint32_t g = gs > NSDO ? gs - NSDO : 0; g < gs; ++g)
    drain_wait(&c->do_full[g % NSDO], (g / NSDO) & 1, p.err);
  for (uint32_t g = gst > NSDO ? gst - NSDO : 0; g < gst; ++g)
    drain_wait(&c->st_full[g % NSDO], (g / NSDO) & 1, p.err);
}

__device__ void mma_role(const BwdParams& p, uint8_t* smem, BsCtl* c, uint32_t tbase) {
  const uint32_t leader = elect_one();
  const uint32_t id_s = idesc_bf16_f32(128, 128, false, false);  // S, dP
  const uint32_t id_q = idesc_bf16_f32(128, D, false, true);     // dQ (A = dS in TMEM)
  const uint32_t id_kv = idesc_bf16_f32(128, D, true, true);     // dV, dK (A, B MN-major)
  const int nks = cdiv(p.Lq, 16);  // K steps of the products over queries
  const uint64_t q_k = smem_desc_sw128(smem_addr(smem + kQ), 16, 1024);
  const uint64_t q_m = smem_desc_sw128(smem_addr(smem + kQ), 16384, 1024);
  const uint64_t do_k0 = smem_desc_sw128(smem_addr(smem + kDO), 16, 1024);
  const uint64_t do_m0 = smem_desc_sw128(smem_addr(smem + kDO), 16384, 1024);
  const uint64_t k_k0 = smem_desc_sw128(smem_addr(smem + kK), 16, 1024);
  const uint64_t k_m0 = smem_desc_sw128(smem_addr(smem + kK), 16384, 1024);
  const uint64_t v_k0 = smem_desc_sw128(smem_addr(smem + kV), 16, 1024);
  const uint64_t pt_m = smem_desc_sw128(smem_addr(smem + kPT), 16384, 1024);
  const uint64_t dst_m = smem_desc_sw128(smem_addr(smem + kDST), 16384, 1024);
  uint32_t itq = 0, nk = 0, nv = 0, gs = 0, gt = 0, gi = 0;
  bool ok = true, issued = false;
  for (uint32_t n = 0; ok; ++n) {
    BsDec f;
    if (!next_item(c, n, &f, &ok, p.err)) break;
    if (f.n == 0) continue;
    if (!mbar_wait_warp(&c->q_full, itq & 1, &c->abort, p.err)) break;
    ++itq;
    const uint32_t k0 = nk, v0 = nv, t0 = gt;
    Seg sg;
    seg_load(sg, p.offsets, p.B, f.b, f.j);
    int st = 0;
    uint64_t do_m = do_m0, do_k = do_k0;
    for (int u = 0; u <= f.n && ok; ++u) {
      if (u >= 1) {
        const uint32_t t = t0 + u - 1;  // global key-tile index of u - 1
        const int buf = t & 1;
        if (!mbar_wait_warp(&c->ds_full, t & 1, &c->abort, p.err)) { ok = false; break; }
        if (u == 1 && !mbar_wait_warp(&c->dq_free, (gi & 1) ^ 1, &c->abort, p.err)) { ok = false; break; }
        tc_fence_after();
        const uint64_t km = desc_add(k_m0, ((k0 + u - 1) % NSK) * kTile);
#pragma unroll
        for (int k = 0; k < kBN / 16; ++k)  // dQ += dS K(u-1): dS packed at SP + 8k (+32 for keys 64..)
          if (leader)
            mma_ts(tbase + kColDQ, tbase + kColSP + 8 * k + (k >= 4 ? 32 : 0),
                   desc_add(km, k * 2048), id_q, (u > 1) || (k > 0));
        if (u == f.n && leader) mma_commit(&c->dq_full);
        for (int k = 0; k < nks; ++k)  // dK = dS^T Q
          if (leader)
            mma_ss(tbase + col_dk(buf), desc_add(dst_m, k * 2048), desc_add(q_m, k * 2048), id_kv,
                   k > 0);
        if (leader) {
          mma_commit(&c->dkdv_full[buf]);
          mma_commit(&c->k_empty[(k0 + u - 1) % NSK]);  // K(u-1): read by S and dQ
        }
        if (u == f.n && leader) mma_commit(&c->q_empty);  // Q: read by S and dK
      }
      if (u < f.n) {
        const uint32_t t = t0 + u;
        const int buf = t & 1;
        const bool seg_start = u == 0 || sg.j == 0;
        const bool seg_end = u == f.n - 1 || sg.j == sg.nts - 1;
        if (seg_start) {
          st = gs % NSDO;
          do_m = desc_add(do_m0, st * kTile);
          do_k = desc_add(do_k0, st * kTile);
        }
        const uint32_t kk = k0 + u;
        if (!mbar_wait_warp(&c->k_full[kk % NSK], (kk / NSK) & 1, &c->abort, p.err)) { ok = false; break; }
        tc_fence_after();
        const uint64_t kk_k = desc_add(k_k0, (kk % NSK) * kTile);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)  // S = Q K^T
          if (leader)
            mma_ss(tbase + kColSP, desc_add(q_k, k * 32), desc_add(kk_k, k * 32), id_s, k > 0);
        if (leader) mma_commit(&c->s_full);
        issued = true;
        const uint32_t vv = v0 + u;
        if (!mbar_wait_warp(&c->v_full[vv % NSV], (vv / NSV) & 1, &c->abort, p.err)) { ok = false; break; }
        if (seg_start &&
            !mbar_wait_warp(&c->do_full[st], (gs / NSDO) & 1, &c->abort, p.err)) { ok = false; break; }
        if (!mbar_wait_warp(&c->p_done, t & 1, &c->abort, p.err)) { ok = false; break; }
        tc_fence_after();
        const uint64_t vk = desc_add(v_k0, (vv % NSV) * kTile);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)  // dP = dO V^T
          if (leader) mma_ss(tbase + kColSP, desc_add(do_k, k * 32), desc_add(vk, k * 32), id_s, k > 0);
        if (leader) {
          mma_commit(&c->dp_full);
          mma_commit(&c->v_empty[vv % NSV]);
        }
        // dV = P^T dO into the buffer of tile t, free once the epilogue of
        // tile t - 2 has read it.
        if (!mbar_wait_warp(&c->p_full, t & 1, &c->abort, p.err)) { ok = false; break; }
        if (!mbar_wait_warp(&c->dkdv_empty[buf], ((t >> 1) & 1) ^ 1, &c->abort, p.err)) { ok = false; break; }
        tc_fence_after();
        for (int k = 0; k < nks; ++k)
          if (leader)
            mma_ss(tbase + col_dv(buf), desc_add(pt_m, k * 2048), desc_add(do_m, k * 2048), id_kv,
                   k > 0);
        if (seg_end) {
          if (leader) mma_commit(&c->do_empty[st]);  // dO: read by dP and dV
          ++gs;
        }
        if (u + 1 < f.n) seg_next(sg, p.offsets, p.B);
      }
    }
    if (!ok) break;
    gt += f.n;
    ++gi;
    nk += f.n;
    nv += f.n;
  }
  if (issued && leader) {
    mma_commit(&c->drain);
    drain_wait(&c->drain, 0, p.err);
  }
}

__device__ void math_role(const BwdParams& p, uint8_t* smem, BsCtl* c, uint32_t tbase) {
  const int r = threadIdx.x & 127;    // TMEM lane: query row (scores), key row (epilogue)
  const int half = threadIdx.x >> 7;  // key columns 64*half.. (scores); dV / dK (epilogue)
  const uint32_t lane_base = static_cast<uint32_t>((r >> 5) * 32) << 16;
  const int T = p.hdr->T;
  const float sl2 = p.scale_log2;
  const uint64_t sl2x2 = f2_pack(sl2, sl2);
  // This thread's 128-byte row of the P^T / dS^T operands: key chunk `half`,
  // query (K index) r; 16-byte unit u at (u ^ (r & 7)) * 16.
  uint8_t* pt_row = smem + kPT + half * kTile + r * 128;
  uint8_t* dst_row = smem + kDST + half * kTile + r * 128;
  uint32_t gt = 0, gi = 0, gs = 0;
  bool ok = true;
  // Epilogue of key tile t: dV (half 0) or scale * dK (half 1) of key row r,
  // stored if the row is a key of the sequence.
  auto epilogue = [&](uint32_t t, int h, int off0, int j, const KvTile& kt) {
    const int buf = t & 1;
    if (!mbar_wait_warp(&c->dkdv_full[buf], (t >> 1) & 1, &c->abort, p.err)) return false;
    tc_fence_after();
    uint32_t a[2][32];
    const uint32_t col = half == 0 ? col_dv(buf) : col_dk(buf);
    tmem_ld32(tbase + lane_base + col, a[0]);
    tmem_ld32(tbase + lane_base + col + 32, a[1]);
    tmem_wait_ld();
    tc_fence_before();
    mbar_arrive(&c->dkdv_empty[buf]);
    const float mul = half == 0 ? 1.f : p.scale;
    uint32_t w[32];
#pragma unroll
    for (int ch = 0; ch < 2; ++ch)
#pragma unroll
      for (int i = 0; i < 16; ++i)
        w[16 * ch + i] = pack_bf16x2(__uint_as_float(a[ch][2 * i]) * mul,
                                     __uint_as_float(a[ch][2 * i + 1]) * mul);
    if (r >= kt.shift && r < kt.shift + kt.nk) {
      const long long tok = static_cast<long long>(off0) + j * kBN - kt.shift + r;
      __nv_bfloat16* dst = (half == 0 ? p.dv : p.dk) + (tok * p.H + h) * D;
      st_global_64B(dst, w);
      st_global_64B(dst + 32, w + 16);
    }
    return true;
  };
  for (uint32_t n = 0; ok; ++n) {
    BsDec f;
    if (!next_item(c, n, &f, &ok, p.err)) break;
    if (f.n == 0) continue;
    uint64_t nlse2 = 0, ndlt2 = 0;
    Seg sg;
    seg_load(sg, p.offsets, p.B, f.b, f.j);
    KvTile prev_kt = {0, 0, 0};
    int prev_off0 = 0, prev_j = 0;
    for (int u = 0; u < f.n && ok; ++u) {
      const uint32_t t = gt + u;
      if (u == 0 || sg.j == 0) {
        const int st = gs % NSDO;
        if (!mbar_wait_warp(&c->st_full[st], (gs / NSDO) & 1, &c->abort, p.err)) { ok = false; break; }
        const float* e = reinterpret_cast<const float*>(smem + kStat + st * kStatBytes) + stat_float(r);
        nlse2 = f2_pack(e[0], e[0]);
        ndlt2 = f2_pack(e[4], e[4]);
        mbar_arrive(&c->st_empty[st]);
        ++gs;
      }
      const KvTile kt = kv_tile(sg.off0, sg.L, sg.j, T);
      // ---- P: S leaves TMEM first (dP may then overwrite SP)
      if (!mbar_wait_warp(&c->s_full, t & 1, &c->abort, p.err)) { ok = false; break; }
      tc_fence_after();
      const uint32_t ts = tbase + lane_base + kColSP + 64 * half;
      uint32_t pk[32];
      {
        uint32_t sraw[2][32];
        tmem_ld32(ts, sraw[0]);
        tmem_ld32(ts + 32, sraw[1]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&c->p_done);
#pragma unroll
        for (int ch = 0; ch < 2; ++ch)
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 x = f2_unpack(ffma2(f2_pack(__uint_as_float(sraw[ch][2 * i]),
                                                     __uint_as_float(sraw[ch][2 * i + 1])),
                                             sl2x2, nlse2));
            pk[16 * ch + i] = pack_bf16x2(ex2_approx(x.x), ex2_approx(x.y));
          }
      }
      if (kt.nk < kBN || kt.shift > 0) {  // keep key columns [shift, shift + nk)
        const int lo = kt.shift - 64 * half;
        const uint32_t span = kt.nk > 0 ? static_cast<uint32_t>(kt.nk) : 0u;
#pragma unroll
        for (int i = 0; i < 32; ++i)
          pk[i] &= (static_cast<uint32_t>(2 * i - lo) < span ? 0x0000ffffu : 0u) |
                   (static_cast<uint32_t>(2 * i + 1 - lo) < span ? 0xffff0000u : 0u);
      }
      // P^T operand row (free: dV of the previous tile completed before S)
#pragma unroll
      for (int q = 0; q < 8; ++q)
        *reinterpret_cast<uint4*>(pt_row + ((q ^ (r & 7)) << 4)) =
            make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      fence_proxy_async_smem();
      mbar_arrive(&c->p_full);
      // ---- dS = P (dP - Delta)
      if (!mbar_wait_warp(&c->dp_full, t & 1, &c->abort, p.err)) { ok = false; break; }
      tc_fence_after();
      uint32_t w[32];
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t praw[32];
        tmem_ld32(ts + 32 * ch, praw);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 d = f2_unpack(fadd2(
              f2_pack(__uint_as_float(praw[2 * i]), __uint_as_float(praw[2 * i + 1])), ndlt2));
          w[16 * ch + i] = bmul2(pk[16 * ch + i], pack_bf16x2(d.x, d.y));
        }
      }
      tmem_st16(ts, *reinterpret_cast<const uint32_t(*)[16]>(w));
      tmem_st16(ts + 16, *reinterpret_cast<const uint32_t(*)[16]>(w + 16));
#pragma unroll
      for (int q = 0; q < 8; ++q)
        *reinterpret_cast<uint4*>(dst_row + ((q ^ (r & 7)) << 4)) =
            make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&c->ds_full);
      // ---- epilogue of the previous key tile, under this tile's products
      if (u >= 1 && !epilogue(t - 1, f.h, prev_off0, prev_j, prev_kt)) { ok = false; break; }
      prev_kt = kt;
      prev_off0 = sg.off0;
      prev_j = sg.j;
      if (u + 1 < f.n) seg_next(sg, p.offsets, p.B);
    }
    if (!ok) break;
    if (!epilogue(gt + f.n - 1, f.h, prev_off0, prev_j, prev_kt)) break;
    gt += f.n;
    // dQ partial (unscaled), rows of the dense Q only: part[slot][0][r][:]
    if (!mbar_wait_warp(&c->dq_full, gi & 1, &c->abort, p.err)) break;
    tc_fence_after();
    {
      uint32_t v[32];
      tmem_ld32(tbase + lane_base + kColDQ + 32 * half, v);
      tmem_wait_ld();
      if (r < p.Lq) {
        float* dst = p.dq_part + (static_cast<long long>(f.slot) * 2 * kBM + r) * D + 32 * half;
#pragma unroll
        for (int q = 0; q < 4; ++q) st_global_v8(dst + 8 * q, v + 8 * q);
      }
    }
    tc_fence_before();
    mbar_arrive(&c->dq_free);
    ++gi;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    bwd_bs_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                  const BwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  BsCtl* c = reinterpret_cast<BsCtl*>(smem + kCtl);
  const int warp = warp_id(), lane = lane_id();
  if ((smem_addr(smem) & 1023) != 0) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrSmemAlign);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(&c->q_full, 1);
    mbar_init(&c->q_empty, 1);
    for (int s = 0; s < NSDO; ++s) {
      mbar_init(&c->do_full[s], 1);
      mbar_init(&c->do_empty[s], 1);
      mbar_init(&c->st_full[s], 1);
      mbar_init(&c->st_empty[s], kMath);
    }
    for (int i = 0; i < NSK; ++i) {
      mbar_init(&c->k_full[i], 1);
      mbar_init(&c->k_empty[i], 1);
    }
    for (int i = 0; i < NSV; ++i) {
      mbar_init(&c->v_full[i], 1);
      mbar_init(&c->v_empty[i], 1);
    }
    mbar_init(&c->s_full, 1);
    mbar_init(&c->p_done, kMath);
    mbar_init(&c->p_full, kMath);
    mbar_init(&c->dp_full, 1);
    mbar_init(&c->ds_full, kMath);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&c->dkdv_full[b], 1);
      mbar_init(&c->dkdv_empty[b], kMath);
      mbar_init(&c->item_full[b], 1);
      mbar_init(&c->item_empty[b], 9);  // 8 math warps + the MMA warp
    }
    mbar_init(&c->dq_full, 1);
    mbar_init(&c->dq_free, kMath);
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
    math_role(p, smem, c, tbase);
  } else if (warp == kProducerWarp) {
    if (lane == 0) producer_role(&tq, &tk, &tv, &tdo, p, smem, c);
  } else {
    mma_role(p, smem, c, tbase);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

}  // namespace

bool bwd_bs_supported(int D_, int Lq) { return D_ == D && Lq >= 1 && Lq <= kBM; }

cudaError_t launch_bwd_bs(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const BwdParams& p, int grid, cudaStream_t s) {
  static_assert(kSmem <= 232448, "shared memory budget");
  static_assert(sizeof(BsCtl) <= 512, "control block");
  if (!bwd_bs_supported(D, p.Lq)) return cudaErrorInvalidValue;
  cudaError_t e =
      cudaFuncSetAttribute(bwd_bs_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  bwd_bs_kernel<<<grid, kThreads, kSmem, s>>>(tq, tk, tv, tdo, p);
  return cudaGetLastError();
}

}  // namespace jfa
