// Self-attention backward, pass 1 of 2: dK and dV for sm_103a.
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
//   P^T  = exp2(S^T * scale*log2e - LSE*log2e), bf16 over S^T's columns
//   dS^T = P^T (dP^T - Delta),                bf16 over dP^T's columns
//   dV  += P^T dO       (TS, B = dO MN-major)
//   dK  += dS^T Q       (TS, B = Q MN-major)
// The score math is split into a P part (needs S^T) and a dS part (needs
// dP^T), and the MMAs of consecutive query tiles are interleaved:
//   dV(g), S(g+1), dK(g), dP(g+1), dV(g+1), ...
// so the P part of tile g+1 runs under dK(g) + dP(g+1) and its dS part under
// dV(g+1) + S(g+2).  S(g+1) / dP(g+1) overwrite P^T(g) / dS^T(g) right after
// the dV / dK MMAs that read them (MMAs of one CTA execute in issue order).
//
// CTA = 10 warps: warps 0-7 score/gradient math (warp w: TMEM lanes
// 32*(w%4).. = key rows, query columns 64*(w/4)..) and the dK/dV epilogue,
// warp 8 TMA producer, warp 9 MMA issuer.
#include "common.cuh"
#include "ptx.cuh"

namespace jfa {
namespace {

constexpr int kThreads = 320;
constexpr int kMath = 256;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;

template <int D>
struct KvCfg {
  static constexpr int NSQ = 2;              // Q / dO ring depth
  static constexpr int kTile = kBM * D * 2;  // bytes of a 128-row bf16 tile
  static constexpr int kSlabs = D / 64;
  static constexpr int kK = 0;
  static constexpr int kV = kTile;
  static constexpr int kQ = 2 * kTile;
  static constexpr int kDO = kQ + NSQ * kTile;
  // {LSE*log2e, Delta} of the 128 query rows of each Q / dO stage
  static constexpr int kStatBytes = kBM * 8;
  static constexpr int kStat = kDO + NSQ * kTile;
  static constexpr int kCtl = kStat + NSQ * kStatBytes;
  static constexpr int kSmem = kCtl + 512;
  static constexpr uint32_t kColS = 0, kColDP = 128;
  static constexpr uint32_t kColDV = 256, kColDK = 256 + D;
};

struct KvCtl {
  uint64_t kv_full, kv_empty;
  uint64_t qdo_full[2], qdo_empty[2];
  uint64_t s_full, dp_full, p_full, ds_full;
  uint64_t dkdv_full, dkdv_empty;
  uint64_t item_full[2], item_empty[2];
  uint64_t drain;
  int item_slot[2];
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

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

struct KvItem {
  int b, h, kb;
  int off0, L;
  RowBox kt;   // keys of this block
  int t0, nt;  // first query tile and count
};

template <bool CAUSAL>
__device__ __forceinline__ KvItem decode(const BwdParams& p, int idx, int T) {
  KvItem f;
  const Item it = p.items[idx];
  f.b = it.x;
  f.h = it.y >> 16;
  f.kb = it.y & 0xffff;
  f.off0 = p.offsets[f.b];
  f.L = p.offsets[f.b + 1] - f.off0;
  f.kt = row_box(f.off0 + f.kb * kBN, f.L - f.kb * kBN, T);
  f.t0 = CAUSAL ? (f.kb * kBN) / kBM : 0;
  f.nt = cdiv(f.L, kBM) - f.t0;
  return f;
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

__device__ __forceinline__ int next_item(KvCtl* c, uint32_t n, bool warp, bool* ok, int* err) {
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
                              KvCtl* c) {
  using C = KvCfg<D>;
  const int n_items = p.hdr->n_items;
  const int T = p.hdr->T;
  uint32_t it = 0, gq = 0;
  bool ok = true;
  for (uint32_t n = 0; ok; ++n) {
    const int slot = n & 1;
    if (!mbar_wait(&c->item_empty[slot], ((n >> 1) & 1) ^ 1, &c->abort, p.err)) break;
    const int idx = atomicAdd(&p.hdr->ticket, 1);
    c->item_slot[slot] = idx < n_items ? idx : -1;
    mbar_arrive(&c->item_full[slot]);
    if (idx >= n_items) break;
    const KvItem f = decode<CAUSAL>(p, idx, T);
    if (!mbar_wait(&c->kv_empty, (it & 1) ^ 1, &c->abort, p.err)) break;
    mbar_arrive_expect_tx(&c->kv_full, 2 * C::kTile);
#pragma unroll
    for (int s = 0; s < C::kSlabs; ++s) {
      tma_load_3d(smem + C::kK + s * 16384, tk, &c->kv_full, s * 64, f.h, f.kt.row);
      tma_load_3d(smem + C::kV + s * 16384, tv, &c->kv_full, s * 64, f.h, f.kt.row);
    }
    ++it;
    for (int i = 0; i < f.nt; ++i) {
      const uint32_t g = gq;
      const int st = g % C::NSQ;
      if (!mbar_wait(&c->qdo_empty[st], ((g / C::NSQ) & 1) ^ 1, &c->abort, p.err)) {
        ok = false;
        break;
      }
      const int t = f.t0 + i;
      const RowBox qb = row_box(f.off0 + t * kBM, f.L - t * kBM, T);
      // Row statistics of the box: from stat if its first entry is 16-byte
      // aligned there, else from the copy shifted by one entry.
      const long long sidx = static_cast<long long>(f.h) * T + qb.row;
      const float2* ssrc = (sidx & 1) ? p.stat_odd + (sidx - 1) : p.stat + sidx;
      mbar_arrive_expect_tx(&c->qdo_full[st], 2 * C::kTile + C::kStatBytes);
      bulk_load(smem + C::kStat + st * C::kStatBytes, ssrc, C::kStatBytes, &c->qdo_full[st]);
#pragma unroll
      for (int s = 0; s < C::kSlabs; ++s) {
        tma_load_3d(smem + C::kQ + st * C::kTile + s * 16384, tq, &c->qdo_full[st], s * 64, f.h,
                    qb.row);
        tma_load_3d(smem + C::kDO + st * C::kTile + s * 16384, tdo, &c->qdo_full[st], s * 64, f.h,
                    qb.row);
      }
      ++gq;
    }
  }
  if (it > 0) drain_wait(&c->kv_full, (it - 1) & 1, p.err);
  for (uint32_t g = gq > C::NSQ ? gq - C::NSQ : 0; g < gq; ++g)
    drain_wait(&c->qdo_full[g % C::NSQ], (g / C::NSQ) & 1, p.err);
}

template <int D, bool CAUSAL>
__device__ void mma_role(const BwdParams& p, uint8_t* smem, KvCtl* c, uint32_t tbase) {
  using C = KvCfg<D>;
  const int T = p.hdr->T;
  // Run by the whole warp; the elected lane issues products and commits.
  const uint32_t leader = elect_one();
  const uint32_t id_st = idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
  const uint32_t id_kv = idesc_bf16_f32(128, D, false, true);     // dV, dK (A in TMEM)
  // Descriptors built once; per tile and K step only adds remain.
  const uint64_t dk_k = smem_desc_sw128(smem_addr(smem + C::kK), 16, 1024);
  const uint64_t dv_k = smem_desc_sw128(smem_addr(smem + C::kV), 16, 1024);
  const uint64_t dq_k0 = smem_desc_sw128(smem_addr(smem + C::kQ), 16, 1024);
  const uint64_t ddo_k0 = smem_desc_sw128(smem_addr(smem + C::kDO), 16, 1024);
  const uint64_t dq_m0 = smem_desc_sw128(smem_addr(smem + C::kQ), 16384, 1024);
  const uint64_t ddo_m0 = smem_desc_sw128(smem_addr(smem + C::kDO), 16384, 1024);
  const uint32_t tS = tbase + C::kColS, tDP = tbase + C::kColDP;
  const uint32_t tDV = tbase + C::kColDV, tDK = tbase + C::kColDK;
  // Each issue function runs `mid` before its group's last product: the
  // wait for the next group then overlaps tensor work still queued (issue
  // blocks while the pipe is full; a wait right after a group would leave it
  // idle for the wait's own latency).
  auto issue_s = [&](uint32_t g, auto&& mid) {
    const uint64_t dq_k = desc_add(dq_k0, (g % C::NSQ) * C::kTile);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      if (k == D / 16 - 1 && !mid()) return false;
      const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
      if (leader) mma_ss(tS, desc_add(dk_k, off), desc_add(dq_k, off), id_st, k > 0);
    }
    return true;
  };
  auto issue_dp = [&](uint32_t g, auto&& mid) {
    const uint64_t ddo_k = desc_add(ddo_k0, (g % C::NSQ) * C::kTile);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      if (k == D / 16 - 1 && !mid()) return false;
      const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
      if (leader) mma_ss(tDP, desc_add(dv_k, off), desc_add(ddo_k, off), id_st, k > 0);
    }
    return true;
  };
  // A operand column of query block k (16 queries): packed P^T / dS^T of
  // queries 0-63 start at +0, of queries 64-127 at +64.
  auto issue_dv = [&](uint32_t g, bool acc, auto&& mid) {
    const uint64_t ddo_m = desc_add(ddo_m0, (g % C::NSQ) * C::kTile);
#pragma unroll
    for (int k = 0; k < kBM / 16; ++k) {
      if (k == kBM / 16 - 1 && !mid()) return false;
      if (leader) mma_ts(tDV, tS + k * 8 + (k >= 4 ? 32 : 0), desc_add(ddo_m, k * 2048), id_kv, acc || (k > 0));
    }
    return true;
  };
  auto issue_dk = [&](uint32_t g, bool acc) {
    const uint64_t dq_m = desc_add(dq_m0, (g % C::NSQ) * C::kTile);
#pragma unroll
    for (int k = 0; k < kBM / 16; ++k)
      if (leader) mma_ts(tDK, tDP + k * 8 + (k >= 4 ? 32 : 0), desc_add(dq_m, k * 2048), id_kv, acc || (k > 0));
  };
  auto none = [] { return true; };
  auto wait_qdo = [&](uint32_t g) {
    return mbar_wait_warp(&c->qdo_full[g % C::NSQ], (g / C::NSQ) & 1, &c->abort, p.err);
  };
  auto wait_p = [&](uint32_t g) { return mbar_wait_warp(&c->p_full, g & 1, &c->abort, p.err); };
  auto wait_ds = [&](uint32_t g) { return mbar_wait_warp(&c->ds_full, g & 1, &c->abort, p.err); };
  uint32_t it = 0, gq = 0;
  bool ok = true, issued = false;
  for (uint32_t n = 0; ok; ++n) {
    const int idx = next_item(c, n, true, &ok, p.err);
    if (idx < 0) break;
    const KvItem f = decode<CAUSAL>(p, idx, T);
    if (!mbar_wait_warp(&c->kv_full, it & 1, &c->abort, p.err)) break;
    const uint32_t g0 = gq;
    if (!wait_qdo(g0)) break;
    tc_fence_after();
    issued = true;
    if (!issue_s(g0, none)) break;
    if (leader) mma_commit(&c->s_full);
    // Inside dP(g0): P^T(g0) ready, and the previous item's epilogue has read
    // the dV / dK accumulators.
    if (!issue_dp(g0, [&] {
          return wait_p(g0) && mbar_wait_warp(&c->dkdv_empty, (it & 1) ^ 1, &c->abort, p.err);
        }))
      break;
    if (leader) mma_commit(&c->dp_full);
    // Order per tile g: dV(g), S(g+1), dK(g), dP(g+1).
    for (int i = 0; i < f.nt; ++i) {
      const uint32_t g = g0 + i;
      const bool more = i + 1 < f.nt;
      tc_fence_after();
      if (!issue_dv(g, i > 0, [&] { return !more || wait_qdo(g + 1); })) { ok = false; break; }
      if (more) {  // S(g+1): its P^T(g) columns were just read by dV(g)
        tc_fence_after();
        if (!issue_s(g + 1, [&] { return wait_ds(g); })) { ok = false; break; }
        if (leader) mma_commit(&c->s_full);
      } else if (!wait_ds(g)) {
        ok = false;
        break;
      }
      tc_fence_after();
      issue_dk(g, i > 0);
      if (leader) mma_commit(&c->qdo_empty[g % C::NSQ]);
      if (more) {  // dP(g+1): its dS^T(g) columns were just read by dK(g)
        if (!issue_dp(g + 1, [&] { return wait_p(g + 1); })) { ok = false; break; }
        if (leader) mma_commit(&c->dp_full);
      }
    }
    if (!ok) break;
    gq += f.nt;
    if (leader) mma_commit(&c->dkdv_full);
    if (leader) mma_commit(&c->kv_empty);
    ++it;
  }
  if (issued && leader) {
    mma_commit(&c->drain);
    drain_wait(&c->drain, 0, p.err);
  }
}

template <int D, bool CAUSAL>
__device__ void math_role(const BwdParams& p, uint8_t* smem, KvCtl* c, uint32_t tbase) {
  using C = KvCfg<D>;
  const int r = threadIdx.x & 127;    // TMEM lane = key row of the block
  const int half = threadIdx.x >> 7;  // query columns [64*half, 64*half + 64)
  const uint32_t lane_base = static_cast<uint32_t>((r >> 5) * 32) << 16;
  const int T = p.hdr->T;
  const float sl2 = p.scale_log2;
  uint32_t it = 0, gq = 0;
  bool ok = true;
  for (uint32_t n = 0; ok; ++n) {
    const int idx = next_item(c, n, true, &ok, p.err);
    if (idx < 0) break;
    const KvItem f = decode<CAUSAL>(p, idx, T);
    const int key = f.kb * kBN - f.kt.shift + r;  // local key index of this lane
    const bool key_ok = r >= f.kt.shift && r < f.kt.shift + f.kt.n;
    for (int i = 0; i < f.nt; ++i, ++gq) {
      const uint32_t g = gq;
      const int t = f.t0 + i;
      const RowBox qb = row_box(f.off0 + t * kBM, f.L - t * kBM, T);
      const int q0 = t * kBM - qb.shift;  // local query index of column 0
      // The statistics arrived with Q / dO of the stage (already complete
      // once S^T is; waited on here for their visibility).
      if (!mbar_wait_warp(&c->qdo_full[g % C::NSQ], (g / C::NSQ) & 1, &c->abort, p.err)) { ok = false; break; }
      // Column c: {LSE*log2e, Delta, and the same of column c+1} at stat4[c/2].
      const float4* stat4 = reinterpret_cast<const float4*>(smem + C::kStat + (g % C::NSQ) * C::kStatBytes);
      // Admissible query columns [lo, hi): the box's rows of the sequence
      // and, causal, the queries at or after this key.
      int lo = qb.shift;
      const int hi = qb.shift + qb.n;
      if (CAUSAL) lo = max(lo, key - q0);
      const bool ragged = qb.shift > 0 || qb.n < kBM;
      const bool mask = ragged || (CAUSAL && __any_sync(0xffffffffu, lo > 64 * half));
      const uint32_t span = hi > lo ? static_cast<uint32_t>(hi - lo) : 0u;
      // ---- P part: P^T = exp2(S^T * scale*log2e - LSE*log2e)
      if (!mbar_wait_warp(&c->s_full, g & 1, &c->abort, p.err)) { ok = false; break; }
      tc_fence_after();
      float pv[64];
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const int cbase = 64 * half + 32 * ch;
        uint32_t sraw[32];
        tmem_ld32(tbase + lane_base + C::kColS + cbase, sraw);
        tmem_wait_ld();
        // Rows of keys outside the sequence are left unmasked: row r of dV
        // and dK depends only on row r of P^T and dS^T, and those rows are
        // never stored.
#pragma unroll
        for (int cc = 0; cc < 32; cc += 2) {
          const float4 st2 = stat4[(cbase + cc) / 2];
          pv[32 * ch + cc] = ex2_approx(fmaf(__uint_as_float(sraw[cc]), sl2, -st2.x));
          pv[32 * ch + cc + 1] = ex2_approx(fmaf(__uint_as_float(sraw[cc + 1]), sl2, -st2.z));
        }
        if (mask) {  // ragged or causal diagonal tile: zero inadmissible columns
#pragma unroll
          for (int cc = 0; cc < 32; ++cc)
            pv[32 * ch + cc] =
                static_cast<uint32_t>(cbase + cc - lo) < span ? pv[32 * ch + cc] : 0.f;
        }
        uint32_t pk[16];
#pragma unroll
        for (int cc = 0; cc < 32; cc += 2) pk[cc / 2] = pack_bf16x2(pv[32 * ch + cc], pv[32 * ch + cc + 1]);
        // bf16 pairs of query columns cbase.. land in packed column
        // 64 * half + 16 * ch: inside this half's own, already read columns.
        tmem_st16(tbase + lane_base + C::kColS + 64 * half + 16 * ch, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&c->p_full);
      // ---- dS part: dS^T = P^T (dP^T - Delta)
      if (!mbar_wait_warp(&c->dp_full, g & 1, &c->abort, p.err)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const int cbase = 64 * half + 32 * ch;
        uint32_t praw[32];
        tmem_ld32(tbase + lane_base + C::kColDP + cbase, praw);
        tmem_wait_ld();
        uint32_t dk[16];
#pragma unroll
        for (int cc = 0; cc < 32; cc += 2) {
          const float4 st2 = stat4[(cbase + cc) / 2];
          const float d0 = pv[32 * ch + cc] * (__uint_as_float(praw[cc]) - st2.y);
          const float d1 = pv[32 * ch + cc + 1] * (__uint_as_float(praw[cc + 1]) - st2.w);
          dk[cc / 2] = pack_bf16x2(d0, d1);
        }
        tmem_st16(tbase + lane_base + C::kColDP + 64 * half + 16 * ch, dk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&c->ds_full);
    }
    if (!ok) break;
    // Item epilogue: dV and scale * dK rows of this K/V block (this warp's
    // half of the head dimension).
    if (!mbar_wait_warp(&c->dkdv_full, it & 1, &c->abort, p.err)) break;
    tc_fence_after();
    const long long row = (static_cast<long long>(f.off0) + key) * p.H + f.h;
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const uint32_t col = which == 0 ? C::kColDV : C::kColDK;
      const float mul = which == 0 ? 1.f : p.scale;
      __nv_bfloat16* dst = (which == 0 ? p.dv : p.dk) + row * D;
#pragma unroll
      for (int ch = 0; ch < D / 64; ++ch) {
        const int dbase = (D / 2) * half + 32 * ch;
        uint32_t v[32];
        tmem_ld32(tbase + lane_base + col + dbase, v);
        tmem_wait_ld();
        uint32_t w[16];
#pragma unroll
        for (int i2 = 0; i2 < 16; ++i2)
          w[i2] = pack_bf16x2(__uint_as_float(v[2 * i2]) * mul, __uint_as_float(v[2 * i2 + 1]) * mul);
        if (key_ok) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + dbase);
          d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
          d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
          d4[2] = make_uint4(w[8], w[9], w[10], w[11]);
          d4[3] = make_uint4(w[12], w[13], w[14], w[15]);
        }
      }
    }
    tc_fence_before();
    mbar_arrive(&c->dkdv_empty);
    ++it;
  }
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kv_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                  const BwdParams p) {
  using C = KvCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  KvCtl* c = reinterpret_cast<KvCtl*>(smem + C::kCtl);
  const int warp = warp_id(), lane = lane_id();
  if ((smem_addr(smem) & 1023) != 0) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrSmemAlign);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(&c->kv_full, 1);
    mbar_init(&c->kv_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c->qdo_full[i], 1);
      mbar_init(&c->qdo_empty[i], 1);
      mbar_init(&c->item_full[i], 1);
      mbar_init(&c->item_empty[i], 9);  // 8 math warps + the MMA warp
    }
    mbar_init(&c->s_full, 1);
    mbar_init(&c->dp_full, 1);
    mbar_init(&c->p_full, kMath);
    mbar_init(&c->ds_full, kMath);
    mbar_init(&c->dkdv_full, 1);
    mbar_init(&c->dkdv_empty, kMath);
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
    math_role<D, CAUSAL>(p, smem, c, tbase);
  } else if (warp == kProducerWarp) {
    if (lane == 0) producer_role<D, CAUSAL>(&tq, &tk, &tv, &tdo, p, smem, c);
  } else {
    mma_role<D, CAUSAL>(p, smem, c, tbase);
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
  using C = KvCfg<D>;
  static_assert(C::kSmem <= 232448, "shared memory budget");
  static_assert(sizeof(KvCtl) <= 512, "control block");
  auto kern = bwd_kv_kernel<D, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, C::kSmem, s>>>(tq, tk, tv, tdo, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_kv(int D, bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
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
