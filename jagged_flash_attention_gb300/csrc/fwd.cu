// Jagged flash attention forward for sm_103a.
//
// Method: "Optimizing Jagged Flash Attention with TLX" (pytorch.org),
// section 2.1 (role-specialised warps; hand-allocated SMEM/TMEM buffers; S
// and P sharing one TMEM allocation while the PV accumulator keeps its own;
// the M dimension split into two groups; persistent CTAs) and section 2.2
// (longest-first scheduling, masks only on the ragged tail tile); per-row
// math from "cuTile Kernels - FMHA Implementation", "Flash Attention
// Algorithm" and "exp2 + flush_to_zero" (online softmax in base 2 with the
// scale folded into one multiply-add).
//
// A work item is (sequence b, head h, pair of 128-row query tiles).  Both
// query tiles share every K/V tile the CTA loads.  CTA = 10 warps, one CTA
// per SM:
//   warps 0-3, 4-7  softmax / correction / epilogue of query tile 0 and 1;
//                   thread r owns row r of its tile (TMEM lane r)
//   warp 8          TMA producer (the two Q tiles once per item, K and V
//                   tiles into rings) and the work scheduling: the grid has
//                   one CTA per possible item; a CTA takes its own item, then
//                   the items of CTAs that have not started, cancelled through
//                   Cluster Launch Control (the TLX page, section 2.2,
//                   "Scheduling jagged tiles across SMs": CLC work stealing
//                   over the precomputed longest-first list)
//   warp 9          TMEM allocation and the tcgen05 issuer (the whole warp
//                   waits; an elect.sync lane issues)
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 and O1 after them.  P_t
// (bf16) overwrites the first 64 columns of S_t and is read from TMEM by the
// PV MMA, in two halves: keys 0-63 are handed over (with any O rescale
// already done) while keys 64-127 are still being written, so PV's first
// four K steps overlap the rest of the softmax.  Issue order per K/V tile j:
// PV0(j-1), S0(j), PV1(j-1), S1(j), so each softmax group has the time of two
// MMAs to turn S into P.  S_t(j) overwrites the columns that PV_t(j-1),
// issued just before it, reads P from; tcgen05 MMAs of one CTA execute in
// issue order.
//
// Variants: with a local mask (causal or a sliding window, the LOCAL
// instantiation) each query tile visits only the key tiles of its band and
// the item streams the union of its two tiles' ranges; with GQA the K/V
// tiles are those of head h / G; the SPARSE instantiation streams the key
// tiles of the item's block list (block-sparse attention).
#include "common.cuh"
#include "ptx.cuh"

namespace jfa {
namespace {

constexpr int kFwdThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr float kLn2 = 0.6931471805599453f;
// Conditional rescaling: the running max used for exp2 is only raised when
// the row max grows by more than 2^kRescaleLog2, so P <= 2^8 and most tiles
// skip the O correction.  The result is exact either way.
constexpr float kRescaleLog2 = 8.f;

template <int D>
struct FwdCfg {
  static constexpr int NSK = (D == 128) ? 3 : 4;  // K ring depth
  static constexpr int NSV = (D == 128) ? 2 : 4;  // V ring depth
  static constexpr int kTile = kBM * D * 2;       // bytes of a 128-row bf16 tile
  static constexpr int kSlabs = D / 64;           // 64-column (128 B) slabs per row
  static constexpr int kQ = 0;                    // two Q tiles
  static constexpr int kK = 2 * kTile;
  static constexpr int kV = kK + NSK * kTile;
  static constexpr int kCtl = kV + NSV * kTile;  // barriers and small state
  static constexpr int kSmem = kCtl + 512;
  __host__ __device__ static constexpr uint32_t colS(int t) { return 128u * t; }
  __host__ __device__ static constexpr uint32_t colO(int t) { return 256u + D * t; }
};


__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

struct QTile {
  int q_lo;   // local index of the tile's first query row
  int nq;     // valid query rows (<= 0: tile absent)
  int shift;  // rows the Q box was moved back to stay inside [0, T)
  int row;    // TMA row coordinate of the Q box
  int j0;     // first key tile this query tile visits
  int n_kv;   // key tiles it visits: [j0, j0 + n_kv)
};

struct FwdItem {
  int b, h, hk;  // sequence, query head, K/V head
  int off0, L;
  QTile t[2];
  int J0, N;  // key tiles loaded for the item: [J0, J0 + N), the union of the tiles' ranges
};

struct FwdCtl {
  uint64_t q_full, q_empty;
  // K stages have one full barrier per 64-column slab ([stage][slab]): S's
  // first K steps need only slab 0.
  uint64_t k_full[4][2], k_empty[4], v_full[4], v_empty[4];
  // P_t in two halves (keys 0-63, 64-127): PV_t's first four K steps start
  // while the softmax writes the second half.
  uint64_t s_full[2], p_half[2], p_full[2], o_ready[2], o_free[2];
  uint64_t item_full[2], item_empty[2];
  uint64_t drain;
  FwdItem item[2];  // decoded by the producer; b < 0: no more items
  uint64_t clc_bar;    // completion of the cluster-launch-control request in flight
  uint4 clc_resp;      // its 16-byte response
  uint32_t tmem_base;
  int abort;
};

// LOCAL: a local mask (causal or a sliding window, bounds p.wl / p.wr): a
// query tile visits only the key tiles that hold admissible keys of its
// rows, and the item streams the union of its two tiles' ranges.
// SPARSE: block-sparse attention (self-attention or broadcast-Q): both query
// tiles of the item visit the key tiles of the item's block list, in its
// (ascending) order; with LOCAL as well (self-attention) the band masks the
// listed tiles, and a row left without an admissible key ends with O = 0,
// LSE = -inf.
template <bool BCAST, bool LOCAL, bool SPARSE>
__device__ __forceinline__ FwdItem decode(const FwdParams& p, int idx, int T) {
  FwdItem f;
  const Item it = p.items[idx];
  f.b = it.x;
  f.h = it.y >> 16;
  f.hk = f.h / p.G;
  const int pair = it.y & 0xffff;
  f.off0 = p.offsets[f.b];
  f.L = p.offsets[f.b + 1] - f.off0;
  int lo = 1 << 30, hi = 0;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    QTile& q = f.t[t];
    q.q_lo = (2 * pair + t) * kBM;
    q.j0 = 0;
    if (BCAST) {
      q.nq = min(kBM, p.Lq - q.q_lo);
      q.shift = 0;
      q.row = q.q_lo;
      q.n_kv = q.nq > 0 ? (SPARSE ? p.counts[(static_cast<long long>(f.b) * p.H + f.h) * p.nqb + pair]
                                  : cdiv(f.L, kBN))
                        : 0;
    } else {
      q.nq = min(kBM, f.L - q.q_lo);
      const int start = f.off0 + q.q_lo;
      q.shift = max(0, start + kBM - T);
      q.row = start - q.shift;
      q.n_kv = 0;
      if (q.nq > 0) {
        if (SPARSE)
          q.n_kv = p.counts[(static_cast<long long>(f.b) * p.H + f.h) * p.nqb + pair];
        else if (LOCAL)
          key_tiles(q.q_lo, q.q_lo + q.nq - 1, f.L, p.wl, p.wr, &q.j0, &q.n_kv);
        else
          q.n_kv = cdiv(f.L, kBN);
      }
    }
    if (q.n_kv > 0) {
      lo = min(lo, q.j0);
      hi = max(hi, q.j0 + q.n_kv);
    }
  }
  f.J0 = hi > 0 ? lo : 0;
  f.N = hi > 0 ? hi - lo : 0;
  return f;
}

// Block list of a sparse item: key tiles in ascending order.
__device__ __forceinline__ const int32_t* sparse_list(const FwdParams& p, const FwdItem& f) {
  const long long row = (static_cast<long long>(f.b) * p.H + f.h) * p.nqb + f.t[0].q_lo / kFwdRows;
  return p.blocks + row * p.kcap;
}

// Key tile of step j of the item's key-tile stream.
template <bool LOCAL, bool SPARSE>
__device__ __forceinline__ int stream_tile(const FwdParams& p, const FwdItem& f, int j) {
  if (SPARSE) return sparse_list(p, f)[j];
  return (LOCAL ? f.J0 : 0) + j;
}

// Key tile j of a sequence: box row coordinate, shift and valid key count.
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

// Wait that ignores the abort flag: used only while draining in-flight
// asynchronous copies and MMAs before the CTA exits.
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
__device__ __forceinline__ bool next_item(FwdCtl* c, uint32_t n, FwdItem* f, bool* ok, int* err) {
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

template <int D, bool LOCAL, bool BCAST, bool SPARSE>
__device__ void producer_role(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                              const FwdParams& p, uint8_t* smem, FwdCtl* c) {
  using C = FwdCfg<D>;
  const int n_items = p.hdr->n_items;
  const int T = p.hdr->T;
  uint32_t itq = 0, nk = 0, nv = 0;
  bool ok = true;
  // Items: this CTA's own index, then the indices of cancelled CTAs.  One
  // request stays in flight while an item runs; after a request finds no CTA
  // left, none is issued again.  Indices past the list (the host sizes the
  // grid by the list's upper bound) only cancel further CTAs.
  uint32_t nclc = 0;     // requests completed
  bool pending = false;  // a request in flight
  auto clc_issue = [&]() {
    mbar_arrive_expect_tx(&c->clc_bar, 16);
    clc_try_cancel(&c->clc_resp, &c->clc_bar);
    pending = true;
  };
  auto clc_take = [&]() {
    if (!pending) return -1;
    pending = false;
    if (!mbar_wait(&c->clc_bar, nclc & 1, &c->abort, p.err)) {
      drain_wait(&c->clc_bar, nclc & 1, p.err);  // the response still lands in shared memory
      ok = false;
      return -1;
    }
    ++nclc;
    int x;
    if (!clc_query(&c->clc_resp, &x)) return -1;
    clc_issue();
    return x;
  };
  int idx = blockIdx.x;
  clc_issue();
  for (uint32_t n = 0; ok; ++n) {
    const int slot = n & 1;
    if (!mbar_wait(&c->item_empty[slot], ((n >> 1) & 1) ^ 1, &c->abort, p.err)) break;
    while (idx >= n_items && ok) idx = clc_take();
    FwdItem f;
    if (idx >= 0 && ok)
      f = decode<BCAST, LOCAL, SPARSE>(p, idx, T);
    else
      f.b = -1;
    c->item[slot] = f;
    mbar_arrive(&c->item_full[slot]);
    if (f.b < 0) break;
    idx = n_items;  // taken: the next index comes from the request in flight
    if (f.N == 0) continue;
    if (!mbar_wait(&c->q_empty, (itq & 1) ^ 1, &c->abort, p.err)) break;
    const int ntl = (f.t[0].n_kv > 0 ? 1 : 0) + (f.t[1].n_kv > 0 ? 1 : 0);
    mbar_arrive_expect_tx(&c->q_full, ntl * C::kTile);
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      if (f.t[t].n_kv == 0) continue;
#pragma unroll
      for (int s = 0; s < C::kSlabs; ++s)
        tma_load_3d(smem + C::kQ + t * C::kTile + s * 16384, tq, &c->q_full, s * 64, f.h,
                    f.t[t].row);
    }
    ++itq;
    // Order K0, K1, V0, K2, V1, ... (of the item's key tiles J0, J0 + 1,
    // ...): the MMA needs K(j) and V(j-1) together.
    for (int j = 0; j <= f.N && ok; ++j) {
      if (j < f.N) {
        const int st = nk % C::NSK;
        const KvTile kt = kv_tile(f.off0, f.L, stream_tile<LOCAL, SPARSE>(p, f, j), T);
        if (!mbar_wait(&c->k_empty[st], ((nk / C::NSK) & 1) ^ 1, &c->abort, p.err)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int s = 0; s < C::kSlabs; ++s) {
          mbar_arrive_expect_tx(&c->k_full[st][s], 16384);
          tma_load_3d(smem + C::kK + st * C::kTile + s * 16384, tk, &c->k_full[st][s], s * 64, f.hk,
                      kt.row);
        }
        ++nk;
      }
      if (j >= 1) {
        const int st = nv % C::NSV;
        const KvTile kt = kv_tile(f.off0, f.L, stream_tile<LOCAL, SPARSE>(p, f, j - 1), T);
        if (!mbar_wait(&c->v_empty[st], ((nv / C::NSV) & 1) ^ 1, &c->abort, p.err)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&c->v_full[st], C::kTile);
#pragma unroll
        for (int s = 0; s < C::kSlabs; ++s)
          tma_load_3d(smem + C::kV + st * C::kTile + s * 16384, tv, &c->v_full[st], s * 64, f.hk,
                      kt.row);
        ++nv;
      }
    }
  }
  // Drain: every copy and request this CTA issued has landed before exit.
  if (pending) drain_wait(&c->clc_bar, nclc & 1, p.err);
  if (itq > 0) drain_wait(&c->q_full, (itq - 1) & 1, p.err);
  for (uint32_t g = nk > C::NSK ? nk - C::NSK : 0; g < nk; ++g)
    for (int s = 0; s < C::kSlabs; ++s) drain_wait(&c->k_full[g % C::NSK][s], (g / C::NSK) & 1, p.err);
  for (uint32_t g = nv > C::NSV ? nv - C::NSV : 0; g < nv; ++g)
    drain_wait(&c->v_full[g % C::NSV], (g / C::NSV) & 1, p.err);
}

// S_t = Q_t K^T, K steps [k0, k1): dq / dk are the K-major descriptors of
// the Q tile and the K stage (start of the tile); K steps advance them inside
// 128-byte rows, step k in 64-column slab k/4.
template <int D>
__device__ __forceinline__ void issue_s(uint32_t leader, uint32_t tbase, int t, uint64_t dq,
                                        uint64_t dk, int k0, int k1) {
  using C = FwdCfg<D>;
  const uint32_t id_s = idesc_bf16_f32(kBM, kBN, false, false);
#pragma unroll
  for (int k = k0; k < k1; ++k) {
    const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
    if (leader) mma_ss(tbase + C::colS(t), desc_add(dq, off), desc_add(dk, off), id_s, k > 0);
  }
}

// O_t += P_t V, K steps [k0, k1) (16 keys each): dv is the MN-major
// descriptor of the V stage.
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t leader, uint32_t tbase, int t, uint64_t dv,
                                         bool accumulate, int k0, int k1) {
  using C = FwdCfg<D>;
  const uint32_t id_pv = idesc_bf16_f32(kBM, D, false, true);
#pragma unroll
  for (int k = k0; k < k1; ++k) {
    if (leader)
      mma_ts(tbase + C::colO(t), tbase + C::colS(t) + k * 8, desc_add(dv, k * 2048), id_pv,
             accumulate || (k > 0));
  }
}

template <int D, bool LOCAL, bool BCAST>
__device__ void mma_role(const FwdParams& p, uint8_t* smem, FwdCtl* c, uint32_t tbase) {
  using C = FwdCfg<D>;
  // Run by the whole warp; the elected lane issues products and commits.
  const uint32_t leader = elect_one();
  const uint64_t dq0 = smem_desc_sw128(smem_addr(smem + C::kQ), 16, 1024);
  const uint64_t dk0 = smem_desc_sw128(smem_addr(smem + C::kK), 16, 1024);
  const uint64_t dv0 = smem_desc_sw128(smem_addr(smem + C::kV), 16384, 1024);
  uint32_t itq = 0, nk = 0, nv = 0;
  uint32_t np[2] = {0, 0};   // P tiles consumed per query tile
  uint32_t ito[2] = {0, 0};  // items per query tile (for o_free)
  bool ok = true;
  bool issued = false;
  for (uint32_t n = 0; ok; ++n) {
    FwdItem f;
    if (!next_item(c, n, &f, &ok, p.err)) break;
    if (f.N == 0) continue;
    if (!mbar_wait_warp(&c->q_full, itq & 1, &c->abort, p.err)) break;
    ++itq;
    for (int j = 0; j <= f.N && ok; ++j) {
      uint64_t dk = 0, dv = 0;
      const int kst = nk % C::NSK;
      const uint32_t kph = (nk / C::NSK) & 1;
      int k_have = 0;  // slabs of K(j) waited for; K is read only by S, after PV_0(j-1)
      if (j < f.N) dk = desc_add(dk0, kst * C::kTile);
      if (j >= 1) {
        const int st = nv % C::NSV;
        if (!mbar_wait_warp(&c->v_full[st], (nv / C::NSV) & 1, &c->abort, p.err)) { ok = false; break; }
        dv = desc_add(dv0, st * C::kTile);
      }
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int nkv = f.t[t].n_kv;
        const int lj = LOCAL ? f.J0 + j - f.t[t].j0 : j;  // step j in query tile t's own key tiles
        if (lj >= 1 && lj - 1 < nkv) {  // O_t += P_t V of the previous step, by halves of P
          if (!mbar_wait_warp(&c->p_half[t], np[t] & 1, &c->abort, p.err)) { ok = false; break; }
          if (lj == 1 && !mbar_wait_warp(&c->o_free[t], (ito[t] & 1) ^ 1, &c->abort, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv<D>(leader, tbase, t, dv, lj > 1, 0, kBN / 32);
          if (!mbar_wait_warp(&c->p_full[t], np[t] & 1, &c->abort, p.err)) { ok = false; break; }
          ++np[t];
          tc_fence_after();
          issue_pv<D>(leader, tbase, t, dv, true, kBN / 32, kBN / 16);
          if (leader) mma_commit(&c->o_ready[t]);
        }
        if (lj >= 0 && lj < nkv && j < f.N) {  // S_t = Q_t K^T, slab 1 of K waited for between its halves
          const uint64_t dq = desc_add(dq0, t * C::kTile);
#pragma unroll
          for (int sl = 0; sl < C::kSlabs; ++sl) {
            if (k_have <= sl) {
              if (!mbar_wait_warp(&c->k_full[kst][sl], kph, &c->abort, p.err)) { ok = false; break; }
              tc_fence_after();
              k_have = sl + 1;
            }
            issue_s<D>(leader, tbase, t, dq, dk, 4 * sl, 4 * sl + 4);
          }
          if (!ok) break;
          if (leader) mma_commit(&c->s_full[t]);
          issued = true;
        }
      }
      if (!ok) break;
      if (j >= 1) {
        if (leader) mma_commit(&c->v_empty[nv % C::NSV]);
        ++nv;
      }
      if (j < f.N) {
        if (leader) mma_commit(&c->k_empty[nk % C::NSK]);
        ++nk;
        if (j == f.N - 1) if (leader) mma_commit(&c->q_empty);
      }
    }
#pragma unroll
    for (int t = 0; t < 2; ++t)
      if (f.t[t].n_kv > 0) ++ito[t];
  }
  if (issued && leader) {
    mma_commit(&c->drain);
    drain_wait(&c->drain, 0, p.err);
  }
}

template <int D, bool LOCAL, bool BCAST, bool SPARSE>
__device__ void softmax_role(const FwdParams& p, FwdCtl* c, uint32_t tbase) {
  using C = FwdCfg<D>;
  const int t = threadIdx.x >> 7;   // query tile of this warpgroup
  const int r = threadIdx.x & 127;  // row of the tile == TMEM lane
  const uint32_t lane_base = static_cast<uint32_t>(((threadIdx.x >> 5) & 3) * 32) << 16;
  const uint32_t ts = tbase + lane_base + C::colS(t);
  const uint32_t to = tbase + lane_base + C::colO(t);
  const int T = p.hdr->T;
  const float sl2 = p.scale_log2;
  const uint64_t sl2x2 = f2_pack(sl2, sl2);
  uint32_t u = 0;  // S tiles of this query tile processed so far (all items)
  bool ok = true;
  for (uint32_t n = 0; ok; ++n) {
    FwdItem f;
    if (!next_item(c, n, &f, &ok, p.err)) break;
    const QTile q = t == 0 ? f.t[0] : f.t[1];  // no dynamic indexing (keeps f in registers)
    if (q.nq <= 0) continue;
    const int qi = q.q_lo - q.shift + r;  // local query index of this row
    const bool row_valid = r >= q.shift && r < q.shift + q.nq;
    __nv_bfloat16* orow;
    float* lrow;
    if (BCAST) {
      orow = p.out + ((static_cast<long long>(f.b) * p.Lq + qi) * p.H + f.h) * D;
      lrow = p.lse + (static_cast<long long>(f.b) * p.H + f.h) * p.Lq + qi;
    } else {
      orow = p.out + ((static_cast<long long>(f.off0) + qi) * p.H + f.h) * D;
      lrow = p.lse + static_cast<long long>(f.h) * T + f.off0 + qi;
    }
    if (q.n_kv == 0) {  // empty broadcast sequence: O = 0, LSE = -inf
      if (row_valid) {
        for (int d = 0; d < D; d += 8) *reinterpret_cast<uint4*>(orow + d) = make_uint4(0, 0, 0, 0);
        *lrow = -INFINITY;
      }
      continue;
    }
    float m_used = -INFINITY, l_run = 0.f;
    const int32_t* lst = SPARSE ? sparse_list(p, f) : nullptr;
    for (int j = 0; j < q.n_kv; ++j, ++u) {
      if (!mbar_wait_warp(&c->s_full[t], u & 1, &c->abort, p.err)) { ok = false; break; }
      tc_fence_after();
      uint32_t raw[4][32];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) tmem_ld32(ts + ch * 32, raw[ch]);
      tmem_wait_ld();
      float s[128];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch)
#pragma unroll
        for (int i = 0; i < 32; ++i) s[ch * 32 + i] = __uint_as_float(raw[ch][i]);
      const int jk = SPARSE ? lst[j] : (LOCAL ? q.j0 + j : j);  // key tile of the sequence
      const KvTile kt = kv_tile(f.off0, f.L, jk, T);
      const int key0 = jk * kBN - kt.shift;  // local key index of column 0
      const int qa = q.q_lo - q.shift;       // local query index of row 0 of the box
      const bool need_mask = kt.nk < kBN || kt.shift > 0 ||
                             (LOCAL && (key0 + kBN - 1 > qa + p.wr || key0 < qa + kBM - 1 - p.wl));
      if (need_mask) {
        // Peeled tail: only the ragged last tile (and, with a local mask,
        // the tiles a band edge crosses) pays for the per-element mask.
        int c_lo = kt.shift, c_hi = kt.shift + kt.nk;
        if (LOCAL) {  // admissible keys [qi - wl, qi + wr]
          c_lo = max(c_lo, qi - p.wl - key0);
          c_hi = min(c_hi, qi + p.wr - key0 + 1);
        }
#pragma unroll
        for (int cc = 0; cc < 128; ++cc) {
          const bool keep = cc >= c_lo && cc < c_hi;
          s[cc] = keep ? s[cc] : -INFINITY;
        }
      }
      // Row max with three-input max: two new columns per instruction, four
      // independent chains.
      float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
      for (int cc = 4; cc < 124; cc += 8) {
        mx0 = fmax3(mx0, s[cc], s[cc + 1]);
        mx1 = fmax3(mx1, s[cc + 2], s[cc + 3]);
        mx2 = fmax3(mx2, s[cc + 4], s[cc + 5]);
        mx3 = fmax3(mx3, s[cc + 6], s[cc + 7]);
      }
      mx0 = fmax3(mx0, s[124], s[125]);
      mx1 = fmax3(mx1, s[126], s[127]);
      const float m_tile = fmax3(fmaxf(mx0, mx1), mx2, mx3) * sl2;
      // Raise the exponent base only when the max grew by more than 2^8.
      const bool raise = m_tile > m_used + kRescaleLog2;
      const float m_new = raise ? m_tile : m_used;
      const float alpha = raise ? ex2_approx(m_used - m_new) : 1.f;
      m_used = m_new;
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const uint64_t negm = f2_pack(-m_use, -m_use);
      uint64_t acc0 = 0, acc1 = 0;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        // 32 columns -> 16 packed bf16 pairs, stored to TMEM right away so
        // that only one chunk of P is live in registers.
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const int cc = ch * 32 + i;
          const float2 x0 = f2_unpack(ffma2(f2_pack(s[cc], s[cc + 1]), sl2x2, negm));
          const float2 x1 = f2_unpack(ffma2(f2_pack(s[cc + 2], s[cc + 3]), sl2x2, negm));
          const float p0 = ex2_approx(x0.x), p1 = ex2_approx(x0.y);
          const float p2 = ex2_approx(x1.x), p3 = ex2_approx(x1.y);
          acc0 = fadd2(acc0, f2_pack(p0, p1));
          acc1 = fadd2(acc1, f2_pack(p2, p3));
          pk[i / 2] = pack_bf16x2(p0, p1);
          pk[i / 2 + 1] = pack_bf16x2(p2, p3);
        }
        tmem_st16(ts + ch * 16, pk);
        if (ch == 1) {
          // Keys 0-63 of P are stored (and their scores dead).  PV of the
          // previous tile was issued before S of this one, so it has
          // completed by now (MMAs complete in issue order): observe it and
          // correct O before the first half of P is handed over.
          if (j > 0) {
            if (!mbar_wait_warp(&c->o_ready[t], (u - 1) & 1, &c->abort, p.err)) { ok = false; break; }
            tc_fence_after();
            if (__any_sync(0xffffffffu, raise)) {
#pragma unroll
              for (int oc = 0; oc < D / 32; ++oc) {
                uint32_t o[32];
                tmem_ld32(to + oc * 32, o);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                tmem_st32(to + oc * 32, o);
              }
            }
          }
          tmem_wait_st();
          tc_fence_before();
          mbar_arrive(&c->p_half[t]);
        }
      }
      if (!ok) break;
      const float2 a0 = f2_unpack(acc0), a1 = f2_unpack(acc1);
      l_run = l_run * alpha + ((a0.x + a0.y) + (a1.x + a1.y));
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&c->p_full[t]);
    }
    if (!ok) break;
    // Epilogue: O / l in bf16 and the natural-log LSE.
    if (!mbar_wait_warp(&c->o_ready[t], (u - 1) & 1, &c->abort, p.err)) break;
    tc_fence_after();
    const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
    for (int ch = 0; ch < D / 32; ++ch) {
      uint32_t o[32];
      tmem_ld32(to + ch * 32, o);
      tmem_wait_ld();
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
      if (row_valid) st_global_64B(orow + ch * 32, w);
    }
    if (row_valid) *lrow = l_run > 0.f ? (m_used + lg2_approx(l_run)) * kLn2 : -INFINITY;
    tc_fence_before();
    mbar_arrive(&c->o_free[t]);
  }
}

template <int D, bool LOCAL, bool BCAST, bool SPARSE>
__global__ void __launch_bounds__(kFwdThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv, const FwdParams p) {
  using C = FwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  FwdCtl* c = reinterpret_cast<FwdCtl*>(smem + C::kCtl);
  const int warp = warp_id(), lane = lane_id();
  if ((smem_addr(smem) & 1023) != 0) {  // TMA/UMMA swizzle atoms need 1 KB alignment
    if (threadIdx.x == 0) atomicOr(p.err, kErrSmemAlign);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(&c->q_full, 1);
    mbar_init(&c->q_empty, 1);
    for (int i = 0; i < C::NSK; ++i) {
      mbar_init(&c->k_full[i][0], 1);
      mbar_init(&c->k_full[i][1], 1);
      mbar_init(&c->k_empty[i], 1);
    }
    for (int i = 0; i < C::NSV; ++i) {
      mbar_init(&c->v_full[i], 1);
      mbar_init(&c->v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c->s_full[i], 1);
      mbar_init(&c->p_half[i], kBM);
      mbar_init(&c->p_full[i], kBM);
      mbar_init(&c->o_ready[i], 1);
      mbar_init(&c->o_free[i], kBM);
      mbar_init(&c->item_full[i], 1);
      mbar_init(&c->item_empty[i], 9);  // 8 softmax warps + the MMA thread
    }
    mbar_init(&c->drain, 1);
    mbar_init(&c->clc_bar, 1);
    c->abort = 0;
    fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
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
    softmax_role<D, LOCAL, BCAST, SPARSE>(p, c, tbase);
  } else if (warp == kProducerWarp) {
    if (lane == 0) producer_role<D, LOCAL, BCAST, SPARSE>(&tq, &tk, &tv, p, smem, c);
  } else {
    mma_role<D, LOCAL, BCAST>(p, smem, c, tbase);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int D, bool LOCAL, bool BCAST, bool SPARSE = false>
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const FwdParams& p, int grid, cudaStream_t s) {
  using C = FwdCfg<D>;
  static_assert(C::kSmem <= 232448, "shared memory budget");
  static_assert(sizeof(FwdCtl) <= 512, "control block");
  static_assert(C::NSK <= 4 && C::NSV <= 4, "ring depth");
  auto kern = fwd_kernel<D, LOCAL, BCAST, SPARSE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kFwdThreads, C::kSmem, s>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int D, bool causal, bool bcast, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const FwdParams& p, int grid, cudaStream_t s,
                       bool sparse) {
  if (sparse) {
    if (causal) {  // a local mask on top of the lists (self-attention only)
      if (bcast) return cudaErrorInvalidValue;
      if (D == 128) return launch_fwd_t<128, true, false, true>(tq, tk, tv, p, grid, s);
      return launch_fwd_t<64, true, false, true>(tq, tk, tv, p, grid, s);
    }
    if (D == 128) {
      if (bcast) return launch_fwd_t<128, false, true, true>(tq, tk, tv, p, grid, s);
      return launch_fwd_t<128, false, false, true>(tq, tk, tv, p, grid, s);
    }
    if (bcast) return launch_fwd_t<64, false, true, true>(tq, tk, tv, p, grid, s);
    return launch_fwd_t<64, false, false, true>(tq, tk, tv, p, grid, s);
  }
  if (D == 128) {
    if (bcast) return launch_fwd_t<128, false, true>(tq, tk, tv, p, grid, s);
    if (causal) return launch_fwd_t<128, true, false>(tq, tk, tv, p, grid, s);
    return launch_fwd_t<128, false, false>(tq, tk, tv, p, grid, s);
  }
  if (bcast) return launch_fwd_t<64, false, true>(tq, tk, tv, p, grid, s);
  if (causal) return launch_fwd_t<64, true, false>(tq, tk, tv, p, grid, s);
  return launch_fwd_t<64, false, false>(tq, tk, tv, p, grid, s);
}

}  // namespace jfa
