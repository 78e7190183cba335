// Jagged flash attention backward for broadcast-Q (dK/dV main loop + dQ
// reduction across the batch) for sm_103a.
//
// Method: "Optimizing Jagged Flash Attention with TLX" (pytorch.org):
//  * "Scheduling jagged tiles across SMs": the backward loops over K/V
//    blocks on the outside and Q tiles on the inside; work items are the
//    valid (sequence, head, K/V block) tiles, block-innermost.
//  * "2-CTA collaborative MMA": five GEMMs per K/V block produce dQ, dK, dV.
//  * section 2.1: a dedicated dQ-reduction role next to the load, MMA and
//    softmax roles; "Multi-stage dQ staging" / "Early tensor-memory
//    release": the dQ partial of every K/V block is summed in fp32 across
//    CTAs (broadcast-Q: across the whole batch, into one of several shards)
//    while the MMA warp already works on the next Q tile.
//  * "Loop peeling": masks cost nothing on interior tiles; invalid query
//    columns are removed through an LSE of +inf and invalid key rows through
//    a per-thread predicate, so only causal diagonal tiles test elements.
//
// Per K/V block (128 keys) and Q tile (128 queries), scores are kept
// transposed (keys on TMEM lanes):
//   S^T  = K Q^T            (SS, K-major / K-major)        -> TMEM [0,128)
//   dP^T = V dO^T           (SS)                           -> TMEM [128,256)
//   P^T  = exp2(S^T * scale*log2e - LSE*log2e) -> TMEM (bf16, over S^T)
//   dS   = P (dP - Delta)                      -> SMEM (bf16, swizzled)
//   dV  += P^T dO           (TS: A = P^T in TMEM, B = dO MN-major)
//   dK  += dS^T Q           (SS: A = dS^T K-major, B = Q MN-major)
//   D=128: dQ^T = K^T dS^T  (SS, both MN-major) -> TMEM [128,256), head dims
//          on lanes so that each warp of the reduction adds whole 128-byte
//          lines of the fp32 accumulator
//   D=64:  dQ = dS K        (SS, both MN-major) -> TMEM [384,448)
// CTA = 10 warps: warps 0-3 score/gradient math and the dK/dV epilogue,
// warps 4-7 dQ reduction, warp 8 TMA producer, warp 9 MMA issuer.
#include "common.cuh"
#include "ptx.cuh"

namespace jfa {
namespace {

constexpr int kBwdThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdCfg {
  static constexpr int NSQ = 2;              // Q / dO ring depth
  static constexpr int kTile = kBM * D * 2;  // bytes of a 128-row bf16 tile
  static constexpr int kSlabs = D / 64;
  static constexpr int kK = 0;
  static constexpr int kV = kTile;
  static constexpr int kQ = 2 * kTile;
  static constexpr int kDO = kQ + NSQ * kTile;
  static constexpr int kDS = kDO + NSQ * kTile;  // dS: [128 keys][128 queries] bf16
  static constexpr int kStat = kDS + 32768;     // LSE*log2e and Delta, 2 buffers
  static constexpr int kCtl = kStat + 2 * 2 * kBM * 4;
  static constexpr int kSmem = kCtl + 512;
  static constexpr uint32_t kColS = 0, kColDP = 128;
  static constexpr uint32_t kColDV = 256, kColDK = 256 + D;
  static constexpr bool kDqT = (D == 128);                  // dQ computed transposed
  static constexpr uint32_t kColDQ = kDqT ? kColDP : 384;  // D=128: reuses dP^T
};

struct BwdCtl {
  uint64_t kv_full, kv_empty;
  uint64_t qdo_full[2], qdo_empty[2];
  uint64_t st_full, ds_full;
  uint64_t dq_full, dq_empty;
  uint64_t dkdv_full, dkdv_empty;
  uint64_t stat_full;  // LSE/Delta of the current Q tile staged by all 128 math threads
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
// 128-row box starting at packed row `start` of a sequence with `remaining`
// rows left; moved back so it never reads past row T.
__device__ __forceinline__ RowBox row_box(int start, int remaining, int T) {
  RowBox r;
  r.shift = max(0, start + 128 - T);
  r.row = start - r.shift;
  r.n = min(128, remaining);
  return r;
}

struct BwdTile {
  int b, h, kb;
  int off0, L;
  RowBox kt;   // keys of this block
  int t0, nt;  // first query tile and count
  int rot;     // the Q tiles are visited starting at t0 + rot (mod nt)
};

template <bool BCAST, bool CAUSAL>
__device__ __forceinline__ BwdTile decode(const BwdParams& p, int idx, int T) {
  BwdTile f;
  const Item it = p.items[idx];
  f.b = it.x;
  f.h = it.y >> 16;
  f.kb = it.y & 0xffff;
  f.off0 = p.offsets[f.b];
  f.L = p.offsets[f.b + 1] - f.off0;
  f.kt = row_box(f.off0 + f.kb * kBN, f.L - f.kb * kBN, T);
  if (BCAST) {
    f.t0 = 0;
    f.nt = cdiv(p.Lq, kBM);
    f.rot = (f.b + f.kb) % f.nt;
  } else {
    f.t0 = CAUSAL ? (f.kb * kBN) / kBM : 0;
    f.nt = cdiv(f.L, kBM) - f.t0;
    // Concurrent K/V blocks of one sequence start on different Q tiles so
    // their dQ additions land on different rows.
    f.rot = CAUSAL ? 0 : f.kb % f.nt;
  }
  return f;
}

__device__ __forceinline__ int q_tile_at(const BwdTile& f, int i) {
  int t = f.rot + i;
  if (t >= f.nt) t -= f.nt;
  return f.t0 + t;
}

// Query tile t of the item: box and valid rows.
template <bool BCAST>
__device__ __forceinline__ RowBox q_box(const BwdParams& p, const BwdTile& f, int t, int T) {
  if (BCAST) {
    RowBox r;
    r.row = t * kBM;
    r.shift = 0;
    r.n = min(kBM, p.Lq - t * kBM);
    return r;
  }
  return row_box(f.off0 + t * kBM, f.L - t * kBM, T);
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

// Item queue consumer: returns the item index or -1 at the end.  `warp`:
// called by a whole warp (lane 0 arrives) rather than by a single thread.
__device__ __forceinline__ int next_item(BwdCtl* c, uint32_t n, bool warp, bool* ok, int* err) {
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

template <int D, bool CAUSAL, bool BCAST>
__device__ void producer_role(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                              const CUtensorMap* tdo, const BwdParams& p, uint8_t* smem,
                              BwdCtl* c) {
  using C = BwdCfg<D>;
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
    const BwdTile f = decode<BCAST, CAUSAL>(p, idx, T);
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
      const int t = q_tile_at(f, i);
      const RowBox qb = q_box<BCAST>(p, f, t, T);
      mbar_arrive_expect_tx(&c->qdo_full[st], 2 * C::kTile);
#pragma unroll
      for (int s = 0; s < C::kSlabs; ++s) {
        tma_load_3d(smem + C::kQ + st * C::kTile + s * 16384, tq, &c->qdo_full[st], s * 64, f.h,
                    qb.row);
        if (BCAST)
          tma_load_4d(smem + C::kDO + st * C::kTile + s * 16384, tdo, &c->qdo_full[st], s * 64,
                      f.h, qb.row, f.b);
        else
          tma_load_3d(smem + C::kDO + st * C::kTile + s * 16384, tdo, &c->qdo_full[st], s * 64,
                      f.h, qb.row);
      }
      ++gq;
    }
  }
  if (it > 0) drain_wait(&c->kv_full, (it - 1) & 1, p.err);
  for (uint32_t g = gq > C::NSQ ? gq - C::NSQ : 0; g < gq; ++g)
    drain_wait(&c->qdo_full[g % C::NSQ], (g / C::NSQ) & 1, p.err);
}

template <int D, bool CAUSAL, bool BCAST>
__device__ void mma_role(const BwdParams& p, uint8_t* smem, BwdCtl* c, uint32_t tbase) {
  using C = BwdCfg<D>;
  // Run by the whole warp; the elected lane issues products and commits.
  const uint32_t leader = elect_one();
  const int T = p.hdr->T;
  const uint32_t id_st = idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
  const uint32_t id_dv = idesc_bf16_f32(128, D, false, true);     // dV (A = P^T in TMEM)
  const uint32_t id_dk = idesc_bf16_f32(128, D, false, true);     // dK (A = dS^T K-major)
  const uint32_t id_dq = C::kDqT ? idesc_bf16_f32(128, 128, true, true)  // dQ^T
                                 : idesc_bf16_f32(128, D, true, true);   // dQ
  // Descriptors built once; per tile and K step only adds remain.
  const uint64_t dk_k = smem_desc_sw128(smem_addr(smem + C::kK), 16, 1024);
  const uint64_t dk_m = smem_desc_sw128(smem_addr(smem + C::kK), 16384, 1024);
  const uint64_t dv_k = smem_desc_sw128(smem_addr(smem + C::kV), 16, 1024);
  const uint64_t dq_k0 = smem_desc_sw128(smem_addr(smem + C::kQ), 16, 1024);
  const uint64_t dq_m0 = smem_desc_sw128(smem_addr(smem + C::kQ), 16384, 1024);
  const uint64_t ddo_k0 = smem_desc_sw128(smem_addr(smem + C::kDO), 16, 1024);
  const uint64_t ddo_m0 = smem_desc_sw128(smem_addr(smem + C::kDO), 16384, 1024);
  const uint64_t dds_k = smem_desc_sw128(smem_addr(smem + C::kDS), 16, 1024);
  const uint64_t dds_m = smem_desc_sw128(smem_addr(smem + C::kDS), 16384, 1024);
  uint32_t it = 0, gq = 0;
  bool ok = true, issued = false;
  for (uint32_t n = 0; ok; ++n) {
    const int idx = next_item(c, n, true, &ok, p.err);
    if (idx < 0) break;
    const BwdTile f = decode<BCAST, CAUSAL>(p, idx, T);
    if (!mbar_wait_warp(&c->kv_full, it & 1, &c->abort, p.err)) break;
    for (int i = 0; i < f.nt; ++i, ++gq) {
      const uint32_t g = gq;
      const int st = g % C::NSQ;
      const uint32_t so = st * C::kTile;
      const uint64_t dq_k = desc_add(dq_k0, so), dq_m = desc_add(dq_m0, so);
      const uint64_t ddo_k = desc_add(ddo_k0, so), ddo_m = desc_add(ddo_m0, so);
      if (!mbar_wait_warp(&c->qdo_full[st], (g / C::NSQ) & 1, &c->abort, p.err)) { ok = false; break; }
      tc_fence_after();
      // S^T overwrites P^T of the previous tile, read by its dV MMA issued
      // earlier (MMAs of one CTA execute in issue order).
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
        if (leader) mma_ss(tbase + C::kColS, desc_add(dk_k, off), desc_add(dq_k, off), id_st, k > 0);
      }
      // D=128: dQ^T of the previous tile lives in the dP^T columns.
      if (C::kDqT && g > 0 && !mbar_wait_warp(&c->dq_empty, (g - 1) & 1, &c->abort, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
        if (leader) mma_ss(tbase + C::kColDP, desc_add(dv_k, off), desc_add(ddo_k, off), id_st, k > 0);
      }
      if (leader) mma_commit(&c->st_full);
      issued = true;
      if (!mbar_wait_warp(&c->ds_full, g & 1, &c->abort, p.err)) { ok = false; break; }
      if (i == 0 && !mbar_wait_warp(&c->dkdv_empty, (it & 1) ^ 1, &c->abort, p.err)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < kBM / 16; ++k)
        if (leader) mma_ts(tbase + C::kColDV, tbase + C::kColS + k * 8, desc_add(ddo_m, k * 2048), id_dv,
               (i > 0) || (k > 0));
#pragma unroll
      for (int k = 0; k < kBM / 16; ++k) {
        const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
        if (leader) mma_ss(tbase + C::kColDK, desc_add(dds_k, off), desc_add(dq_m, k * 2048), id_dk,
               (i > 0) || (k > 0));
      }
      if (leader) mma_commit(&c->qdo_empty[st]);
      if (!C::kDqT && g > 0 && !mbar_wait_warp(&c->dq_empty, (g - 1) & 1, &c->abort, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < kBN / 16; ++k) {
        if (!leader) continue;
        if (C::kDqT)
          mma_ss(tbase + C::kColDQ, desc_add(dk_m, k * 2048), desc_add(dds_m, k * 2048), id_dq,
                 k > 0);
        else
          mma_ss(tbase + C::kColDQ, desc_add(dds_m, k * 2048), desc_add(dk_m, k * 2048), id_dq,
                 k > 0);
      }
      if (leader) mma_commit(&c->dq_full);
    }
    if (!ok) break;
    if (leader) mma_commit(&c->dkdv_full);
    if (leader) mma_commit(&c->kv_empty);
    ++it;
  }
  if (issued && leader) {
    mma_commit(&c->drain);
    drain_wait(&c->drain, 0, p.err);
  }
}

template <int D, bool CAUSAL, bool BCAST>
__device__ void math_role(const BwdParams& p, uint8_t* smem, BwdCtl* c, uint32_t tbase) {
  using C = BwdCfg<D>;
  const int r = threadIdx.x;  // TMEM lane = key row of the block
  const int warp = r >> 5;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  const int T = p.hdr->T;
  const float sl2 = p.scale_log2;
  float* s_lse = reinterpret_cast<float*>(smem + C::kStat);  // [2][128]
  float* s_dlt = s_lse + 2 * kBM;                            // [2][128]
  uint8_t* sds = smem + C::kDS;
  uint32_t it = 0, gq = 0;
  bool ok = true;
  for (uint32_t n = 0; ok; ++n) {
    const int idx = next_item(c, n, true, &ok, p.err);
    if (idx < 0) break;
    const BwdTile f = decode<BCAST, CAUSAL>(p, idx, T);
    const int key = f.kb * kBN - f.kt.shift + r;  // local key index of this lane
    const bool key_ok = r >= f.kt.shift && r < f.kt.shift + f.kt.n;
    for (int i = 0; i < f.nt; ++i, ++gq) {
      const uint32_t g = gq;
      const int t = q_tile_at(f, i);
      const RowBox qb = q_box<BCAST>(p, f, t, T);
      const int q0 = t * kBM - qb.shift;  // local query index of column 0
      // Stage LSE*log2e and Delta of this Q tile's rows (thread r: row r).
      {
        const int qi = q0 + r;
        const bool q_ok = r >= qb.shift && r < qb.shift + qb.n;
        float lv = INFINITY, dv = 0.f;
        if (q_ok) {
          const long long si = BCAST ? (static_cast<long long>(f.b) * p.H + f.h) * p.Lq + qi
                                     : static_cast<long long>(f.h) * T + f.off0 + qi;
          lv = p.lse[si] * kLog2e;
          dv = p.delta[si];
        }
        s_lse[(g & 1) * kBM + r] = lv;
        s_dlt[(g & 1) * kBM + r] = dv;
      }
      mbar_arrive(&c->stat_full);
      if (!mbar_wait_warp(&c->stat_full, g & 1, &c->abort, p.err)) { ok = false; break; }
      const float* lse_t = s_lse + (g & 1) * kBM;
      const float* dlt_t = s_dlt + (g & 1) * kBM;
      if (!mbar_wait_warp(&c->st_full, g & 1, &c->abort, p.err)) { ok = false; break; }
      tc_fence_after();
      // Causal: key > query is masked; column c is admissible iff c >= c_min.
      const int c_min = CAUSAL ? key - q0 : -1;
      const bool diag = CAUSAL && __any_sync(0xffffffffu, c_min > 0);
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t sraw[32], praw[32];
        tmem_ld32(tbase + lane_base + C::kColS + ch * 32, sraw);
        tmem_ld32(tbase + lane_base + C::kColDP + ch * 32, praw);
        tmem_wait_ld();
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int cc = 0; cc < 32; cc += 2) {
          const int col = ch * 32 + cc;
          float p0 = ex2_approx(fmaf(__uint_as_float(sraw[cc]), sl2, -lse_t[col]));
          float p1 = ex2_approx(fmaf(__uint_as_float(sraw[cc + 1]), sl2, -lse_t[col + 1]));
          if (!key_ok) p0 = 0.f, p1 = 0.f;
          if (diag) {
            p0 = col >= c_min ? p0 : 0.f;
            p1 = col + 1 >= c_min ? p1 : 0.f;
          }
          const float d0 = p0 * (__uint_as_float(praw[cc]) - dlt_t[col]);
          const float d1 = p1 * (__uint_as_float(praw[cc + 1]) - dlt_t[col + 1]);
          pk[cc / 2] = pack_bf16x2(p0, p1);
          dk[cc / 2] = pack_bf16x2(d0, d1);
        }
        tmem_st16(tbase + lane_base + C::kColS + ch * 16, pk);
        // dS row r (queries ch*32 .. ch*32+31) into the swizzled SMEM tile.
        uint8_t* slab = sds + (ch >> 1) * 16384 + r * 128;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int unit = (ch & 1) * 4 + u;
          *reinterpret_cast<uint4*>(slab + ((unit ^ (r & 7)) << 4)) =
              make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
        }
      }
      tmem_wait_st();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&c->ds_full);
    }
    if (!ok) break;
    // Item epilogue: dV and scale * dK rows of this K/V block.
    if (!mbar_wait_warp(&c->dkdv_full, it & 1, &c->abort, p.err)) break;
    tc_fence_after();
    const long long row = (static_cast<long long>(f.off0) + key) * p.H + f.h;
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const uint32_t col = which == 0 ? C::kColDV : C::kColDK;
      const float mul = which == 0 ? 1.f : p.scale;
      __nv_bfloat16* dst = (which == 0 ? p.dv : p.dk) + row * D;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t v[32];
        tmem_ld32(tbase + lane_base + col + ch * 32, v);
        tmem_wait_ld();
        uint32_t w[16];
#pragma unroll
        for (int i2 = 0; i2 < 16; ++i2)
          w[i2] = pack_bf16x2(__uint_as_float(v[2 * i2]) * mul, __uint_as_float(v[2 * i2 + 1]) * mul);
        if (key_ok) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + ch * 32);
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

// dQ reduction role (warps 4-7): drains each Q tile's dQ partial from TMEM
// into the fp32 accumulator while the other roles move on.
template <int D, bool CAUSAL, bool BCAST>
__device__ void dq_role(const BwdParams& p, BwdCtl* c, uint32_t tbase) {
  using C = BwdCfg<D>;
  const int r = threadIdx.x - 128;  // TMEM lane
  const uint32_t lane_base = static_cast<uint32_t>((r >> 5) * 32) << 16;
  const int T = p.hdr->T;
  const int shard = BCAST ? static_cast<int>(blockIdx.x % p.dq_shards) : 0;
  float* acc = p.dq_acc + (BCAST ? shard * p.shard_stride : 0);
  uint32_t gq = 0;
  bool ok = true;
  for (uint32_t n = 0; ok; ++n) {
    const int idx = next_item(c, n, true, &ok, p.err);
    if (idx < 0) break;
    const BwdTile f = decode<BCAST, CAUSAL>(p, idx, T);
    for (int i = 0; i < f.nt; ++i, ++gq) {
      const uint32_t g = gq;
      const int t = q_tile_at(f, i);
      const RowBox qb = q_box<BCAST>(p, f, t, T);
      const int q0 = t * kBM - qb.shift;  // local query index of column / lane 0
      // Row (query) index into the accumulator for local query qi.
      const long long rbase = BCAST ? 0 : f.off0;
      if (!mbar_wait_warp(&c->dq_full, g & 1, &c->abort, p.err)) { ok = false; break; }
      tc_fence_after();
      if (C::kDqT) {
        // Lane r holds head dim r of every query column: each warp adds 32
        // consecutive floats (one 128-byte line) per query row.
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t v[32];
          tmem_ld32(tbase + lane_base + C::kColDQ + ch * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int cc = 0; cc < 32; ++cc) {
            const int col = ch * 32 + cc;
            if (col >= qb.shift && col < qb.shift + qb.n) {  // warp-uniform
              float* dst = acc + ((rbase + q0 + col) * p.H + f.h) * D + r;
              atomicAdd(dst, __uint_as_float(v[cc]));
            }
          }
        }
      } else {
        // Lane r holds query row r: 16-byte vector additions along the row.
        const bool q_ok = r >= qb.shift && r < qb.shift + qb.n;
        float* dst = acc + ((rbase + q0 + r) * p.H + f.h) * D;
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t v[32];
          tmem_ld32(tbase + lane_base + C::kColDQ + ch * 32, v);
          tmem_wait_ld();
          if (q_ok) {
#pragma unroll
            for (int u = 0; u < 8; ++u)
              atomicAdd(reinterpret_cast<float4*>(dst + ch * 32 + 4 * u),
                        make_float4(__uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1]),
                                    __uint_as_float(v[4 * u + 2]), __uint_as_float(v[4 * u + 3])));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&c->dq_empty);
    }
  }
}

template <int D, bool CAUSAL, bool BCAST>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
               const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  BwdCtl* c = reinterpret_cast<BwdCtl*>(smem + C::kCtl);
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
      mbar_init(&c->item_empty[i], 9);  // 4 math + 4 dQ warps + the MMA thread
    }
    mbar_init(&c->st_full, 1);
    mbar_init(&c->ds_full, kBM);
    mbar_init(&c->dq_full, 1);
    mbar_init(&c->dq_empty, kBM);
    mbar_init(&c->dkdv_full, 1);
    mbar_init(&c->dkdv_empty, kBM);
    mbar_init(&c->stat_full, kBM);
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
  if (warp < 4) {
    math_role<D, CAUSAL, BCAST>(p, smem, c, tbase);
  } else if (warp < 8) {
    dq_role<D, CAUSAL, BCAST>(p, c, tbase);
  } else if (warp == kProducerWarp) {
    if (lane == 0) producer_role<D, CAUSAL, BCAST>(&tq, &tk, &tv, &tdo, p, smem, c);
  } else {
    mma_role<D, CAUSAL, BCAST>(p, smem, c, tbase);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int D, bool CAUSAL, bool BCAST>
cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const BwdParams& p, int grid, cudaStream_t s) {
  using C = BwdCfg<D>;
  static_assert(C::kSmem <= 232448, "shared memory budget");
  static_assert(sizeof(BwdCtl) <= 512, "control block");
  auto kern = bwd_kernel<D, CAUSAL, BCAST>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kBwdThreads, C::kSmem, s>>>(tq, tk, tv, tdo, p);
  return cudaGetLastError();
}

}  // namespace

// Broadcast-Q backward (self-attention uses the two-pass kernels of
// bwd_kv.cu and bwd_q.cu, which need no dQ accumulator).
cudaError_t launch_bwd(int D, bool causal, bool bcast, const CUtensorMap& tq,
                       const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                       const BwdParams& p, int grid, cudaStream_t s) {
  if (!bcast || causal) return cudaErrorInvalidValue;
  if (D == 128) return launch_bwd_t<128, false, true>(tq, tk, tv, tdo, p, grid, s);
  return launch_bwd_t<64, false, true>(tq, tk, tv, tdo, p, grid, s);
}

}  // namespace jfa
