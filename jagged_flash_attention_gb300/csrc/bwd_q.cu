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
//          into SP's first 64 columns
//   dQ  += dS K_j       (TS, B = K MN-major)  -> TMEM DQ
// Each item is a pair of 128-row query tiles of one (sequence, head) that
// share every K / V tile.  The two tiles ping-pong: math warpgroup g owns
// tile g, and the MMA issuer interleaves
//   dQ_0(j-1) S_0(j) | dQ_1(j-1) S_1(j) | dP_0(j) | dP_1(j)
// so that one tile's score math runs under the other tile's products.  One
// chain per tile (S -> P math -> dP -> dS math -> dQ) has several hand-offs
// of a few hundred cycles each; with a single tile in flight the tensor pipe
// idles for most of every chain.
//
// TMEM (512 columns): tile g uses SP at 256g (128 fp32 columns) and DQ at
// 256g + 128 (D columns).  SMEM: Q and dO of both tiles, a K ring and a V
// ring (D = 128: 128 + 64 + 32 KB).
//
// CTA = 10 warps: warpgroup g = warps 4g..4g+3 (thread = query row of tile
// g, all 128 key columns) does tile g's math and its dQ epilogue, warp 8 is
// the TMA producer, warp 9 the MMA issuer.
#include "common.cuh"
#include "ptx.cuh"

namespace jfa {
namespace {

constexpr int kThreads = 320;
constexpr int kGroup = 128;  // threads of one math warpgroup
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr float kLog2e = 1.4426950408889634f;

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

struct QCtl {
  uint64_t qdo_full, qdo_empty;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], p_done[2], dp_full[2], ds_full[2];  // per query tile
  uint64_t dq_full[2], dq_free[2];
  uint64_t item_full[2], item_empty[2];
  uint64_t drain;
  int item_slot[2];
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

struct QTile {
  int q_lo;   // local index of the tile's first query row
  int nq;     // valid query rows (<= 0: tile absent)
  int shift;  // rows the box was moved back to stay inside [0, T)
  int row;    // TMA row coordinate
  int n;      // key tiles this query tile visits (0: absent)
};

struct QItem {
  int b, h, off0, L;
  int N;  // key tiles of the item = max over its two query tiles
  QTile t[2];
};

template <bool CAUSAL>
__device__ __forceinline__ QItem decode(const BwdParams& p, int idx, int T) {
  QItem f;
  const Item it = p.items[idx];
  f.b = it.x;
  f.h = it.y >> 16;
  const int pair = it.y & 0xffff;
  f.off0 = p.offsets[f.b];
  f.L = p.offsets[f.b + 1] - f.off0;
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    QTile& q = f.t[g];
    q.q_lo = (2 * pair + g) * kBM;
    q.nq = min(kBM, f.L - q.q_lo);
    const int start = f.off0 + q.q_lo;
    q.shift = max(0, start + kBM - T);
    q.row = start - q.shift;
    q.n = q.nq > 0 ? (CAUSAL ? cdiv(q.q_lo + q.nq, kBN) : cdiv(f.L, kBN)) : 0;
  }
  f.N = max(f.t[0].n, f.t[1].n);
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

__device__ __forceinline__ int next_item(QCtl* c, uint32_t n, bool warp, bool* ok, int* err) {
  const int slot = n & 1;
  const bool got = warp ? mbar_wait_warp(&c->item_full[slot], (n >> 1) & 1, &c->abort, err)
                        : mbar_wait(&c->item_full[slot], (n >> 1) & 1, &c->abort, err);
  if (!got) {
    *ok = false;
    return -1;
  }
  const int idx = c->item_slot[slot];
  if (warp) __syncwarp();
  if (!warp || (threadIdx.x & 31) == 0) mbar_arrive(&c->item_empty[slot]);
  return idx;
}

template <int D, bool CAUSAL>
__device__ void producer_role(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                              const CUtensorMap* tdo, const BwdParams& p, uint8_t* smem,
                              QCtl* c) {
  using C = QCfg<D>;
  const int n_items = p.hdr->n_items;
  const int T = p.hdr->T;
  uint32_t it = 0, nk = 0, nv = 0;
  bool ok = true;
  for (uint32_t n = 0; ok; ++n) {
    const int slot = n & 1;
    if (!mbar_wait(&c->item_empty[slot], ((n >> 1) & 1) ^ 1, &c->abort, p.err)) break;
    const int idx = atomicAdd(&p.hdr->ticket, 1);
    c->item_slot[slot] = idx < n_items ? idx : -1;
    mbar_arrive(&c->item_full[slot]);
    if (idx >= n_items) break;
    const QItem f = decode<CAUSAL>(p, idx, T);
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
      const KvTile kt = kv_tile(f.off0, f.L, j, T);
      {
        const int st = nk % C::NSK;
        if (!mbar_wait(&c->k_empty[st], ((nk / C::NSK) & 1) ^ 1, &c->abort, p.err)) { ok = false; break; }
        mbar_arrive_expect_tx(&c->k_full[st], C::kTile);
#pragma unroll
        for (int s = 0; s < C::kSlabs; ++s)
          tma_load_3d(smem + C::kK + st * C::kTile + s * 16384, tk, &c->k_full[st], s * 64, f.h,
                      kt.row);
        ++nk;
      }
      {
        const int st = nv % C::NSV;
        if (!mbar_wait(&c->v_empty[st], ((nv / C::NSV) & 1) ^ 1, &c->abort, p.err)) { ok = false; break; }
        mbar_arrive_expect_tx(&c->v_full[st], C::kTile);
#pragma unroll
        for (int s = 0; s < C::kSlabs; ++s)
          tma_load_3d(smem + C::kV + st * C::kTile + s * 16384, tv, &c->v_full[st], s * 64, f.h,
                      kt.row);
        ++nv;
      }
    }
  }
  if (it > 0) drain_wait(&c->qdo_full, (it - 1) & 1, p.err);
  for (uint32_t g = nk > C::NSK ? nk - C::NSK : 0; g < nk; ++g)
    drain_wait(&c->k_full[g % C::NSK], (g / C::NSK) & 1, p.err);
  for (uint32_t g = nv > C::NSV ? nv - C::NSV : 0; g < nv; ++g)
    drain_wait(&c->v_full[g % C::NSV], (g / C::NSV) & 1, p.err);
}

template <int D, bool CAUSAL>
__device__ void mma_role(const BwdParams& p, uint8_t* smem, QCtl* c, uint32_t tbase) {
  using C = QCfg<D>;
  const int T = p.hdr->T;
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
      mma_ss(tbase + 256 * g, desc_add(dq, off), desc_add(dk, off), id_s, k > 0);
    }
  };
  auto issue_dp = [&](int g, uint32_t vidx) {
    const uint64_t ddo = desc_add(dq_k0, (2 * g + 1) * C::kTile);
    const uint64_t dv = desc_add(dv_k0, (vidx % C::NSV) * C::kTile);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
      mma_ss(tbase + 256 * g, desc_add(ddo, off), desc_add(dv, off), id_s, k > 0);
    }
  };
  auto issue_dq = [&](int g, uint32_t kidx, bool acc) {
    // A = dS, bf16 pairs of key columns packed in SP's columns [0, 64).
    const uint64_t dk = desc_add(dk_m0, (kidx % C::NSK) * C::kTile);
#pragma unroll
    for (int k = 0; k < kBN / 16; ++k)
      mma_ts(tbase + 256 * g + 128, tbase + 256 * g + 8 * k, desc_add(dk, k * 2048), id_dq,
             acc || (k > 0));
  };
  uint32_t it = 0, nk = 0, nv = 0;
  uint32_t gt[2] = {0, 0};  // tiles processed per query tile slot, over all items
  uint32_t gi[2] = {0, 0};  // items in which the slot was present
  bool ok = true, issued = false;
  for (uint32_t n = 0; ok; ++n) {
    const int idx = next_item(c, n, false, &ok, p.err);
    if (idx < 0) break;
    const QItem f = decode<CAUSAL>(p, idx, T);
    if (!mbar_wait(&c->qdo_full, it & 1, &c->abort, p.err)) break;
    const int N = f.N;
    const int nt[2] = {f.t[0].n, f.t[1].n};
    const uint32_t k0 = nk, v0 = nv;
    // Step j: dQ_g(j-1) and S_g(j) for both tiles, then dP_0(j), dP_1(j).
    for (int j = 0; j <= N && ok; ++j) {
      bool k_ready = false;
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        if (j >= 1 && j - 1 < nt[g]) {
          const uint32_t u = gt[g] + j - 1;
          if (!mbar_wait(&c->ds_full[g], u & 1, &c->abort, p.err)) { ok = false; break; }
          if (j == 1 && !mbar_wait(&c->dq_free[g], (gi[g] & 1) ^ 1, &c->abort, p.err)) { ok = false; break; }
          tc_fence_after();
          issue_dq(g, k0 + j - 1, j > 1);
          if (j == nt[g]) mma_commit(&c->dq_full[g]);
        }
        if (j < nt[g]) {
          if (!k_ready) {
            const uint32_t kk = k0 + j;
            if (!mbar_wait(&c->k_full[kk % C::NSK], (kk / C::NSK) & 1, &c->abort, p.err)) { ok = false; break; }
            k_ready = true;
          }
          tc_fence_after();
          issue_s(g, k0 + j);
          mma_commit(&c->s_full[g]);
          issued = true;
        }
      }
      if (!ok) break;
      if (j >= 1) mma_commit(&c->k_empty[(k0 + j - 1) % C::NSK]);  // K(j-1) fully read
      if (j < N) {
        const uint32_t vv = v0 + j;
        if (!mbar_wait(&c->v_full[vv % C::NSV], (vv / C::NSV) & 1, &c->abort, p.err)) { ok = false; break; }
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          if (j < nt[g]) {
            if (!mbar_wait(&c->p_done[g], (gt[g] + j) & 1, &c->abort, p.err)) { ok = false; break; }
            tc_fence_after();
            issue_dp(g, vv);
            mma_commit(&c->dp_full[g]);
          }
        }
        if (!ok) break;
        mma_commit(&c->v_empty[vv % C::NSV]);
        if (j == N - 1) mma_commit(&c->qdo_empty);  // Q and dO are read by S and dP only
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
  if (issued) {
    mma_commit(&c->drain);
    drain_wait(&c->drain, 0, p.err);
  }
}

template <int D, bool CAUSAL>
__device__ void math_role(const BwdParams& p, QCtl* c, uint32_t tbase) {
  const int g = threadIdx.x >> 7;     // query tile of the item this warpgroup owns
  const int r = threadIdx.x & 127;    // query row of the tile == TMEM lane
  const uint32_t lane_base = static_cast<uint32_t>((r >> 5) * 32) << 16;
  const uint32_t tsp = tbase + lane_base + 256 * g;
  const uint32_t tdq = tsp + 128;
  const int T = p.hdr->T;
  const float sl2 = p.scale_log2;
  uint32_t u = 0, ic = 0;
  bool ok = true;
  for (uint32_t n = 0; ok; ++n) {
    const int idx = next_item(c, n, true, &ok, p.err);
    if (idx < 0) break;
    const QItem f = decode<CAUSAL>(p, idx, T);
    const QTile q = g == 0 ? f.t[0] : f.t[1];
    if (q.n == 0) continue;
    const int qi = q.q_lo - q.shift + r;  // local query index of this row
    const bool row_valid = r >= q.shift && r < q.shift + q.nq;
    float lse2 = INFINITY, dlt = 0.f;  // rows outside the sequence: P = 0
    if (row_valid) {
      const long long si = static_cast<long long>(f.h) * T + f.off0 + qi;
      lse2 = p.lse[si] * kLog2e;
      dlt = p.delta[si];
    }
    const uint64_t sl2x2 = f2_pack(sl2, sl2), nlse2 = f2_pack(-lse2, -lse2);
    const uint64_t ndlt2 = f2_pack(-dlt, -dlt);
    for (int j = 0; j < q.n; ++j, ++u) {
      const KvTile kt = kv_tile(f.off0, f.L, j, T);
      const int key0 = j * kBN - kt.shift;  // local key index of column 0
      const bool need_mask =
          kt.nk < kBN || kt.shift > 0 || (CAUSAL && key0 + kBN - 1 > q.q_lo - q.shift);
      // Admissible key columns of this row: [c_lo, c_lo + span]; an empty
      // range moves c_lo past every column.
      const int c_last = CAUSAL ? min(kt.shift + kt.nk - 1, qi - key0) : kt.shift + kt.nk - 1;
      const int c_lo = c_last >= kt.shift ? kt.shift : kBN;
      const uint32_t span = c_last >= kt.shift ? static_cast<uint32_t>(c_last - kt.shift) : 0u;
      // ---- P = exp2(S * scale*log2e - LSE*log2e), kept as bf16 pairs
      if (!mbar_wait_warp(&c->s_full[g], u & 1, &c->abort, p.err)) { ok = false; break; }
      tc_fence_after();
      uint32_t pk[64];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t sraw[32];
        tmem_ld32(tsp + 32 * ch, sraw);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float2 x = f2_unpack(ffma2(
              f2_pack(__uint_as_float(sraw[2 * i]), __uint_as_float(sraw[2 * i + 1])), sl2x2, nlse2));
          pk[16 * ch + i] = pack_bf16x2(ex2_approx(x.x), ex2_approx(x.y));
        }
        if (need_mask) {  // ragged or diagonal tile: zero the inadmissible columns
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int col = 32 * ch + 2 * i;
            const uint32_t keep =
                (static_cast<uint32_t>(col - c_lo) <= span ? 0x0000ffffu : 0u) |
                (static_cast<uint32_t>(col + 1 - c_lo) <= span ? 0xffff0000u : 0u);
            pk[16 * ch + i] &= keep;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&c->p_done[g]);  // S read: dP may overwrite SP
      // ---- dS = P (dP - Delta), bf16 pairs into SP's columns [0, 64)
      if (!mbar_wait_warp(&c->dp_full[g], u & 1, &c->abort, p.err)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t praw[32];
        tmem_ld32(tsp + 32 * ch, praw);
        tmem_wait_ld();
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          // (dP - Delta) in fp32, rounded to bf16, times the bf16 P.
          const float2 t = f2_unpack(fadd2(
              f2_pack(__uint_as_float(praw[2 * i]), __uint_as_float(praw[2 * i + 1])), ndlt2));
          w[i] = bmul2(pk[16 * ch + i], pack_bf16x2(t.x, t.y));
        }
        // Packed columns [16ch, 16ch + 16) lie in dP columns this thread has
        // already read (chunks 0 .. ch).
        tmem_st16(tsp + 16 * ch, w);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&c->ds_full[g]);
    }
    if (!ok) break;
    // Epilogue: dQ = scale * acc in bf16.
    if (!mbar_wait_warp(&c->dq_full[g], ic & 1, &c->abort, p.err)) break;
    tc_fence_after();
    __nv_bfloat16* dst = p.dq + ((static_cast<long long>(f.off0) + qi) * p.H + f.h) * D;
#pragma unroll
    for (int ch = 0; ch < D / 32; ++ch) {
      uint32_t v[32];
      tmem_ld32(tdq + 32 * ch, v);
      tmem_wait_ld();
      uint32_t w[16];
#pragma unroll
      for (int i2 = 0; i2 < 16; ++i2)
        w[i2] = pack_bf16x2(__uint_as_float(v[2 * i2]) * p.scale,
                            __uint_as_float(v[2 * i2 + 1]) * p.scale);
      if (row_valid) {
        uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * ch);
        d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
        d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
        d4[2] = make_uint4(w[8], w[9], w[10], w[11]);
        d4[3] = make_uint4(w[12], w[13], w[14], w[15]);
      }
    }
    tc_fence_before();
    mbar_arrive(&c->dq_free[g]);
    ++ic;
  }
}

template <int D, bool CAUSAL>
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
      mbar_init(&c->p_done[g], kGroup);
      mbar_init(&c->dp_full[g], 1);
      mbar_init(&c->ds_full[g], kGroup);
      mbar_init(&c->dq_full[g], 1);
      mbar_init(&c->dq_free[g], kGroup);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c->item_full[i], 1);
      mbar_init(&c->item_empty[i], 9);  // 8 math warps + the MMA thread
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
    math_role<D, CAUSAL>(p, c, tbase);
  } else if (warp == kProducerWarp) {
    if (lane == 0) producer_role<D, CAUSAL>(&tq, &tk, &tv, &tdo, p, smem, c);
  } else {
    if (lane == 0) mma_role<D, CAUSAL>(p, smem, c, tbase);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int D, bool CAUSAL>
cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     const CUtensorMap& tdo, const BwdParams& p, int grid, cudaStream_t s) {
  using C = QCfg<D>;
  static_assert(C::kSmem <= 232448, "shared memory budget");
  static_assert(sizeof(QCtl) <= 512, "control block");
  static_assert(C::NSK <= 4 && C::NSV <= 4, "ring depth");
  static_assert(128 + D <= 256, "TMEM columns per query tile");
  auto kern = bwd_q_kernel<D, CAUSAL>;
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
