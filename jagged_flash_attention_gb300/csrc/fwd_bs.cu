// Broadcast-Q forward with a short dense Q (q_len <= 128) for sm_103a,
// streamed over the key tiles of all sequences.
//
// In broadcast-Q mode ("Optimizing Jagged Flash Attention with TLX",
// section 1) every sequence attends with the same dense Q.  When that Q is a
// single 128-row tile, an item is a chunk of the concatenated key-tile
// stream of all sequences (the dQ-pass chunks of the backward): the CTA
// keeps Q in shared memory and streams K and V, the online softmax ("cuTile
// Kernels - FMHA Implementation", "Flash Attention Algorithm"; base 2 with
// the scale folded in) restarts at every sequence boundary, and each
// sequence segment of the chunk ends with its O / LSE epilogue, run by its
// own warpgroup on the other of two O accumulators while the next segment
// computes.  Short sequences therefore cost neither a Q load nor a pipeline
// drain.  A sequence cut by a chunk boundary (the TLX page's long-sequence
// tail, section 2.2, "Scheduling jagged tiles across SMs") is split-KV: each
// piece leaves its normalised O and base-2 LSE as an fp32 partial, and the
// combine kernel merges the pieces with LSE weights.
//
// Per key tile u: S(u) = Q K_u^T (SS) into S[u % NSB]; P = exp2(S * scale *
// log2e - m) in bf16 over S's first 64 columns; O[seg % 2] += P V_u (TS).
// Issue order: S(u) | PV(u - NSB + 1): with three S buffers (D = 64) S runs
// two tiles ahead of PV, so the softmax never waits for its next S behind
// the previous tile's PV.
//
// q_len <= 64 uses the spread layout (softmax_spread): the queries sit in
// rows 0-15 of each 32-row lane quadrant of the tile, so that the softmax of
// the rows that count runs on all four SM sub-partitions.
//
// CTA = 4 * SPLIT + 6 warps (SPLIT = 2: a four-way split measured slower,
// the softmax being bound by latency rather than by its element count): warps
// 0 .. 4*SPLIT-1 softmax (thread: query row r = TMEM lane, key columns
// (128 / SPLIT) * (warp / 4)..; the SPLIT threads of a row exchange their
// partial row max through shared memory each tile, so all apply the same
// running max), then four epilogue warps for finished segments, the TMA
// producer warp and the MMA issuer warp.  TMEM: S buffers at 128 * i, then
// O0 and O1 (D columns each).
#include "common.cuh"
#include "ptx.cuh"

namespace jfa {
namespace {

// Column split of the softmax, warps and threads of the CTA.
template <int D>
struct FsRoles {
  static constexpr int SPLIT = 2;
  static constexpr int kCols = kBN / SPLIT;        // key columns per softmax thread
  static constexpr int kSoftmax = kBM * SPLIT;     // softmax threads
  static constexpr int kEpiWarp = 4 * SPLIT;       // first epilogue warp
  static constexpr int kProducerWarp = kEpiWarp + 4;
  static constexpr int kMmaWarp = kEpiWarp + 5;
  static constexpr int kThreads = 32 * (kEpiWarp + 6);
};
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleLog2 = 8.f;  // raise the running max only past 2^8 (exact either way)

template <int D>
struct FsCfg {
  static constexpr int NSK = (D == 128) ? 3 : 4;
  static constexpr int NSV = (D == 128) ? 2 : 4;
  static constexpr int kTile = kBM * D * 2;
  static constexpr int kSlabs = D / 64;
  static constexpr int kQ = 0;
  static constexpr int kK = kTile;
  static constexpr int kV = kK + NSK * kTile;
  // (m, l) per row and column part, two segment parities
  static constexpr int kSeg = kV + NSV * kTile;
  // partial row max per row and column part, two tile parities
  static constexpr int kXch = kSeg + 2 * FsRoles<D>::SPLIT * kBM * 8;
  static constexpr int kCtl = kXch + 2 * FsRoles<D>::SPLIT * kBM * 4;
  static constexpr int kSmem = kCtl + 512;
  static constexpr int NSB = (D == 64) ? 3 : 2;  // S buffers: 128 * NSB + 2 * D <= 512 columns
  __host__ __device__ static constexpr uint32_t colS(int i) { return 128u * i; }
  __host__ __device__ static constexpr uint32_t colO(int par) { return 128u * NSB + D * par; }
};

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

struct FsDec {
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

struct FsCtl {
  uint64_t q_full, q_empty;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[3], p_full[3], o_ready[2];  // o_ready[t % 2]: PV(t) complete
  uint64_t o_done[2], o_free[2], seg_full[2], seg_empty[2];
  uint64_t xbar[2];  // the row-max exchange of tile t, t % 2
  uint64_t item_full[2], item_empty[2];
  uint64_t drain;
  FsDec item[2];
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

__device__ __forceinline__ bool next_item(FsCtl* c, uint32_t n, FsDec* f, bool* ok, int* err) {
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

// SPREAD: the Q map's box is 16 rows, and query rows [16 k, 16 k + 16) go to
// tile rows [32 k, 32 k + 16) (the other rows are never read as queries).
template <int D, bool SPREAD>
__device__ void producer_role(const CUtensorMap* tq, const CUtensorMap* tk, const CUtensorMap* tv,
                              const FwdParams& p, uint8_t* smem, FsCtl* c) {
  using C = FsCfg<D>;
  const int n_items = p.hdr->n_items;
  const int T = p.hdr->T;
  uint32_t itq = 0, nk = 0, nv = 0;
  bool ok = true;
  for (uint32_t n = 0; ok; ++n) {
    const int slot = n & 1;
    if (!mbar_wait(&c->item_empty[slot], ((n >> 1) & 1) ^ 1, &c->abort, p.err)) break;
    const int idx = atomicAdd(&p.hdr->ticket, 1);
    FsDec f;
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
    if (SPREAD) {
      const int nbox = min(4, cdiv(p.Lq, 16));
      mbar_arrive_expect_tx(&c->q_full, nbox * C::kSlabs * 16 * 128);
      for (int k = 0; k < nbox; ++k)
#pragma unroll
        for (int s = 0; s < C::kSlabs; ++s)
          tma_load_3d(smem + C::kQ + s * 16384 + k * 32 * 128, tq, &c->q_full, s * 64, f.h, 16 * k);
    } else {
      mbar_arrive_expect_tx(&c->q_full, C::kTile);
#pragma unroll
      for (int s = 0; s < C::kSlabs; ++s)
        tma_load_3d(smem + C::kQ + s * 16384, tq, &c->q_full, s * 64, f.h, 0);
    }
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
  if (itq > 0) drain_wait(&c->q_full, (itq - 1) & 1, p.err);
  for (uint32_t g = nk > C::NSK ? nk - C::NSK : 0; g < nk; ++g)
    drain_wait(&c->k_full[g % C::NSK], (g / C::NSK) & 1, p.err);
  for (uint32_t g = nv > C::NSV ? nv - C::NSV : 0; g < nv; ++g)
    drain_wait(&c->v_full[g % C::NSV], (g / C::NSV) & 1, p.err);
}

template <int D>
__device__ void mma_role(const FwdParams& p, uint8_t* smem, FsCtl* c, uint32_t tbase) {
  using C = FsCfg<D>;
  const uint32_t leader = elect_one();
  const uint32_t id_s = idesc_bf16_f32(kBM, kBN, false, false);
  const uint32_t id_pv = idesc_bf16_f32(kBM, D, false, true);
  const uint64_t dq0 = smem_desc_sw128(smem_addr(smem + C::kQ), 16, 1024);
  const uint64_t dk0 = smem_desc_sw128(smem_addr(smem + C::kK), 16, 1024);
  const uint64_t dv0 = smem_desc_sw128(smem_addr(smem + C::kV), 16384, 1024);
  uint32_t itq = 0, nk = 0, nv = 0, g = 0, gseg = 0;
  bool ok = true, issued = false;
  for (uint32_t n = 0; ok; ++n) {
    FsDec f;
    if (!next_item(c, n, &f, &ok, p.err)) break;
    if (f.n == 0) continue;
    if (!mbar_wait_warp(&c->q_full, itq & 1, &c->abort, p.err)) break;
    ++itq;
    // S runs LA tiles ahead of PV; the cursor follows the PV stream.
    constexpr int LA = C::NSB - 1;
    Seg sg;
    seg_load(sg, p.offsets, p.B, f.b, f.j);
    for (int u = 0; u < f.n + LA && ok; ++u) {
      if (u < f.n) {  // S(u) = Q K_u^T into S[(g + u) % NSB]
        const uint32_t kk = nk + u;
        const int sb = (g + u) % C::NSB;
        if (!mbar_wait_warp(&c->k_full[kk % C::NSK], (kk / C::NSK) & 1, &c->abort, p.err)) { ok = false; break; }
        tc_fence_after();
        const uint64_t dk = desc_add(dk0, (kk % C::NSK) * C::kTile);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
          if (leader) mma_ss(tbase + C::colS(sb), desc_add(dq0, off), desc_add(dk, off), id_s, k > 0);
        }
        if (leader) {
          mma_commit(&c->s_full[sb]);
          mma_commit(&c->k_empty[kk % C::NSK]);  // K is read by S only
          if (u == f.n - 1) mma_commit(&c->q_empty);
        }
        issued = true;
      }
      if (u >= LA) {  // O[seg % 2] += P(v) V_v, v = u - LA
        const int v = u - LA;
        const bool start = v == 0 || sg.j == 0;
        const bool end = v == f.n - 1 || sg.j == sg.nts - 1;
        const uint32_t t = g + v;
        const uint32_t vv = nv + v;
        const int par = gseg & 1;
        if (!mbar_wait_warp(&c->p_full[t % C::NSB], (t / C::NSB) & 1, &c->abort, p.err)) { ok = false; break; }
        if (!mbar_wait_warp(&c->v_full[vv % C::NSV], (vv / C::NSV) & 1, &c->abort, p.err)) { ok = false; break; }
        if (start &&
            !mbar_wait_warp(&c->o_free[par], ((gseg >> 1) & 1) ^ 1, &c->abort, p.err)) { ok = false; break; }
        tc_fence_after();
        const uint64_t dv = desc_add(dv0, (vv % C::NSV) * C::kTile);
#pragma unroll
        for (int k = 0; k < kBN / 16; ++k)
          if (leader)
            mma_ts(tbase + C::colO(par), tbase + C::colS(t % C::NSB) + k * 8,
                   desc_add(dv, k * 2048), id_pv, !start || k > 0);
        if (leader) {
          mma_commit(&c->o_ready[t & 1]);
          mma_commit(&c->v_empty[vv % C::NSV]);
          if (end) mma_commit(&c->o_done[par]);
        }
        if (end) ++gseg;
        if (v + 1 < f.n) seg_next(sg, p.offsets, p.B);
      }
    }
    if (!ok) break;
    g += f.n;
    nk += f.n;
    nv += f.n;
  }
  if (issued && leader) {
    mma_commit(&c->drain);
    drain_wait(&c->drain, 0, p.err);
  }
}

template <int D>
__device__ void softmax_role(const FwdParams& p, uint8_t* smem, FsCtl* c, uint32_t tbase) {
  using C = FsCfg<D>;
  using R = FsRoles<D>;
  constexpr int NC = R::kCols;        // key columns of this thread
  const int r = threadIdx.x & 127;    // query row == TMEM lane
  const int part = threadIdx.x >> 7;  // key columns [NC * part, NC * part + NC)
  const uint32_t lane_base = static_cast<uint32_t>((r >> 5) * 32) << 16;
  const int T = p.hdr->T;
  const float sl2 = p.scale_log2;
  const uint64_t sl2x2 = f2_pack(sl2, sl2);
  float2* seg_ml = reinterpret_cast<float2*>(smem + C::kSeg);  // [parity][part][row] = (m, l)
  float* xch = reinterpret_cast<float*>(smem + C::kXch);       // [tile parity][part][row]
  uint32_t g = 0, gseg = 0;
  bool ok = true;
  for (uint32_t n = 0; ok; ++n) {
    FsDec f;
    if (!next_item(c, n, &f, &ok, p.err)) break;
    if (f.n == 0) continue;
    Seg sg;
    seg_load(sg, p.offsets, p.B, f.b, f.j);
    float m_used = -INFINITY, l_run = 0.f;  // l_run: this thread's columns
    for (int u = 0; u < f.n && ok; ++u) {
      const uint32_t t = g + u;
      const bool start = u == 0 || sg.j == 0;
      const bool end = u == f.n - 1 || sg.j == sg.nts - 1;
      if (start) {
        m_used = -INFINITY;
        l_run = 0.f;
      }
      if (!mbar_wait_warp(&c->s_full[t % C::NSB], (t / C::NSB) & 1, &c->abort, p.err)) { ok = false; break; }
      tc_fence_after();
      const uint32_t ts = tbase + lane_base + C::colS(t % C::NSB);
      uint32_t raw[NC];
#pragma unroll
      for (int ch = 0; ch < NC / 32; ++ch)
        tmem_ld32(ts + NC * part + 32 * ch, *reinterpret_cast<uint32_t(*)[32]>(raw + 32 * ch));
      tmem_wait_ld();
      float s[NC];
#pragma unroll
      for (int i = 0; i < NC; ++i) s[i] = __uint_as_float(raw[i]);
      const KvTile kt = kv_tile(sg.off0, sg.L, sg.j, T);
      if (kt.nk < kBN || kt.shift > 0) {  // ragged key tile: columns [shift, shift + nk)
        const int c0 = NC * part;
#pragma unroll
        for (int cc = 0; cc < NC; ++cc)
          s[cc] = (c0 + cc >= kt.shift && c0 + cc < kt.shift + kt.nk) ? s[cc] : -INFINITY;
      }
      float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
      for (int cc = 4; cc < NC - 4; cc += 8) {
        mx0 = fmax3(mx0, s[cc], s[cc + 1]);
        mx1 = fmax3(mx1, s[cc + 2], s[cc + 3]);
        mx2 = fmax3(mx2, s[cc + 4], s[cc + 5]);
        mx3 = fmax3(mx3, s[cc + 6], s[cc + 7]);
      }
      mx0 = fmax3(mx0, s[NC - 4], s[NC - 3]);
      mx1 = fmax3(mx1, s[NC - 2], s[NC - 1]);
      float mx = fmax3(fmaxf(mx0, mx1), mx2, mx3);
      // Exchange with the other parts of the row.  Every softmax thread has
      // read its S columns before arriving, so the P writes below (part q
      // packs into S columns NC/2 * q.., read by another part) come after
      // all reads.
      float* xt = xch + (t & 1) * R::SPLIT * kBM;
      xt[part * kBM + r] = mx;
      tc_fence_before();
      mbar_arrive(&c->xbar[t & 1]);
      if (!mbar_wait_warp(&c->xbar[t & 1], (t >> 1) & 1, &c->abort, p.err)) { ok = false; break; }
      tc_fence_after();
#pragma unroll
      for (int q = 1; q < R::SPLIT; ++q) mx = fmaxf(mx, xt[((part + q) % R::SPLIT) * kBM + r]);
      const float m_tile = mx * sl2;
      const bool raise = m_tile > m_used + kRescaleLog2;
      const float m_new = raise ? m_tile : m_used;
      const float alpha = raise ? ex2_approx(m_used - m_new) : 1.f;
      m_used = m_new;
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const uint64_t negm = f2_pack(-m_use, -m_use);
      uint64_t acc0 = 0, acc1 = 0;
#pragma unroll
      for (int ch = 0; ch < NC / 32; ++ch) {
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
        // keys NC*part + 32ch.. -> packed columns NC/2*part + 16ch..
        tmem_st16(ts + (NC / 2) * part + ch * 16, pk);
      }
      const float2 a0 = f2_unpack(acc0), a1 = f2_unpack(acc1);
      l_run = l_run * alpha + ((a0.x + a0.y) + (a1.x + a1.y));
      if (!start && __any_sync(0xffffffffu, raise)) {
        // A row raised its max: once PV(t - 1) has landed in this segment's
        // O, scale this thread's O columns.  Only these tiles wait for the
        // previous product; the per-parity barrier cannot run two phases
        // ahead of this wait, since PV(t + 1) needs this tile's P first.
        if (!mbar_wait_warp(&c->o_ready[(t - 1) & 1], ((t - 1) >> 1) & 1, &c->abort, p.err)) { ok = false; break; }
        tc_fence_after();
        constexpr int OC = D / R::SPLIT;  // O columns of this thread: 16 or 64
        const uint32_t to = tbase + lane_base + C::colO(gseg & 1) + OC * part;
#pragma unroll
        for (int ch = 0; ch < OC / 16; ++ch) {
          uint32_t o[16];
          tmem_ld16(to + ch * 16, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st16(to + ch * 16, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&c->p_full[t % C::NSB]);
      if (end) {  // hand the segment's (m, l of these columns) to the epilogue warpgroup
        const int par = gseg & 1;
        if (!mbar_wait_warp(&c->seg_empty[par], ((gseg >> 1) & 1) ^ 1, &c->abort, p.err)) { ok = false; break; }
        seg_ml[(par * R::SPLIT + part) * kBM + r] = make_float2(m_used, l_run);
        mbar_arrive(&c->seg_full[par]);
        ++gseg;
      }
      if (u + 1 < f.n) seg_next(sg, p.offsets, p.B);
    }
    if (!ok) break;
    g += f.n;
  }
}

// Softmax of the spread layout (q_len <= 64): query i sits at tile row
// 32 * (i / 16) + i % 16, so that the valid rows fill lanes 0-15 of all four
// TMEM lane quadrants and every sub-partition's warps work on them.  Warp w
// takes quadrant w % 4 and key columns [64 * (w / 4), + 64); through the
// 16-lane load shapes thread t holds rows t/4 and t/4 + 8 of its quadrant,
// two adjacent key columns in every eight, so P packs into bf16 pairs in
// place and four threads share a row (row max and sum over two shuffles).
template <int D>
__device__ void softmax_spread(const FwdParams& p, uint8_t* smem, FsCtl* c, uint32_t tbase) {
  using C = FsCfg<D>;
  using R = FsRoles<D>;
  static_assert(R::SPLIT == 2, "two key-column halves");
  const int warp = threadIdx.x >> 5, ln = threadIdx.x & 31;
  const int quad = warp & 3, part = warp >> 2;
  const int r0 = 32 * quad + (ln >> 2), r1 = r0 + 8;  // tile rows (TMEM lanes) of this thread
  const int cq = 2 * (ln & 3);                         // its first column in every eight
  const bool active = 16 * quad < p.Lq;                // the quadrant holds queries (warp-uniform)
  const uint32_t lane_base = static_cast<uint32_t>(32 * quad) << 16;
  const int T = p.hdr->T;
  const float sl2 = p.scale_log2;
  const uint64_t sl2x2 = f2_pack(sl2, sl2);
  float2* seg_ml = reinterpret_cast<float2*>(smem + C::kSeg);  // [parity][part][row] = (m, l)
  float* xch = reinterpret_cast<float*>(smem + C::kXch);       // [tile parity][part][row]
  uint32_t g = 0, gseg = 0;
  bool ok = true;
  for (uint32_t n = 0; ok; ++n) {
    FsDec f;
    if (!next_item(c, n, &f, &ok, p.err)) break;
    if (f.n == 0) continue;
    Seg sg;
    seg_load(sg, p.offsets, p.B, f.b, f.j);
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // rows r0, r1; l: this thread's columns
    for (int u = 0; u < f.n && ok; ++u) {
      const uint32_t t = g + u;
      const bool start = u == 0 || sg.j == 0;
      const bool end = u == f.n - 1 || sg.j == sg.nts - 1;
      if (start) {
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
      }
      if (!mbar_wait_warp(&c->s_full[t % C::NSB], (t / C::NSB) & 1, &c->abort, p.err)) { ok = false; break; }
      tc_fence_after();
      const uint32_t ts = tbase + lane_base + C::colS(t % C::NSB);
      // s[4i + e]: e = 0, 1 row r0 and e = 2, 3 row r1, key columns
      // 64 * part + 8 i + cq + (e & 1)
      float s[32];
      float mx0 = -INFINITY, mx1 = -INFINITY;
      if (active) {
        uint32_t raw[32];
        tmem_ld_16x256b_x8(ts + 64 * part, raw);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) s[i] = __uint_as_float(raw[i]);
        const KvTile kt = kv_tile(sg.off0, sg.L, sg.j, T);
        if (kt.nk < kBN || kt.shift > 0) {  // ragged key tile: columns [shift, shift + nk)
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int col = 64 * part + 8 * (i >> 2) + cq + (i & 1);
            s[i] = (col >= kt.shift && col < kt.shift + kt.nk) ? s[i] : -INFINITY;
          }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          mx0 = fmax3(mx0, s[4 * i], s[4 * i + 1]);
          mx1 = fmax3(mx1, s[4 * i + 2], s[4 * i + 3]);
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      }
      // Exchange with the other column half.  Every softmax thread has read
      // its S columns before arriving, so the P writes below (half q packs
      // into S columns 32 q.., read by half 0) come after all reads.
      float* xt = xch + (t & 1) * R::SPLIT * kBM;
      if (active && (ln & 3) == 0) {
        xt[part * kBM + r0] = mx0;
        xt[part * kBM + r1] = mx1;
      }
      tc_fence_before();
      mbar_arrive(&c->xbar[t & 1]);
      if (!mbar_wait_warp(&c->xbar[t & 1], (t >> 1) & 1, &c->abort, p.err)) { ok = false; break; }
      tc_fence_after();
      if (active) {
        mx0 = fmaxf(mx0, xt[(1 - part) * kBM + r0]);
        mx1 = fmaxf(mx1, xt[(1 - part) * kBM + r1]);
        const float mt0 = mx0 * sl2, mt1 = mx1 * sl2;
        const bool raise0 = mt0 > m0 + kRescaleLog2, raise1 = mt1 > m1 + kRescaleLog2;
        const float mn0 = raise0 ? mt0 : m0, mn1 = raise1 ? mt1 : m1;
        const float alpha0 = raise0 ? ex2_approx(m0 - mn0) : 1.f;
        const float alpha1 = raise1 ? ex2_approx(m1 - mn1) : 1.f;
        m0 = mn0;
        m1 = mn1;
        const float mu0 = (mn0 == -INFINITY) ? 0.f : mn0, mu1 = (mn1 == -INFINITY) ? 0.f : mn1;
        const uint64_t negm0 = f2_pack(-mu0, -mu0), negm1 = f2_pack(-mu1, -mu1);
        uint64_t acc0 = 0, acc1 = 0;
        uint32_t pk[16];  // 16x128b: pk[2 i] row r0, pk[2 i + 1] row r1, packed column 4 i + t % 4
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 xa = f2_unpack(ffma2(f2_pack(s[4 * i], s[4 * i + 1]), sl2x2, negm0));
          const float2 xb = f2_unpack(ffma2(f2_pack(s[4 * i + 2], s[4 * i + 3]), sl2x2, negm1));
          const float pa = ex2_approx(xa.x), pb = ex2_approx(xa.y);
          const float pc = ex2_approx(xb.x), pd = ex2_approx(xb.y);
          acc0 = fadd2(acc0, f2_pack(pa, pb));
          acc1 = fadd2(acc1, f2_pack(pc, pd));
          pk[2 * i] = pack_bf16x2(pa, pb);
          pk[2 * i + 1] = pack_bf16x2(pc, pd);
        }
        // keys 64 * part.. -> packed columns 32 * part..
        tmem_st_16x128b_x8(ts + 32 * part, pk);
        const float2 a0 = f2_unpack(acc0), a1 = f2_unpack(acc1);
        l0 = l0 * alpha0 + (a0.x + a0.y);
        l1 = l1 * alpha1 + (a1.x + a1.y);
        if (!start && __any_sync(0xffffffffu, raise0 || raise1)) {
          // A row raised its max: once PV(t - 1) has landed in this segment's
          // O, scale this thread's O entries (rows r0, r1; columns of this
          // half).  The per-parity barrier cannot run two phases ahead of
          // this wait, since PV(t + 1) needs this tile's P first.
          if (!mbar_wait_warp(&c->o_ready[(t - 1) & 1], ((t - 1) >> 1) & 1, &c->abort, p.err)) { ok = false; break; }
          tc_fence_after();
          const uint32_t to = tbase + lane_base + C::colO(gseg & 1) + (D / 2) * part;
          if (D == 64) {
            uint32_t o[16];
            tmem_ld_16x256b_x4(to, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i)
              o[i] = __float_as_uint(__uint_as_float(o[i]) * ((i & 2) ? alpha1 : alpha0));
            tmem_st_16x256b_x4(to, o);
          } else {
            uint32_t o[32];
            tmem_ld_16x256b_x8(to, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              o[i] = __float_as_uint(__uint_as_float(o[i]) * ((i & 2) ? alpha1 : alpha0));
            tmem_st_16x256b_x8(to, o);
          }
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&c->p_full[t % C::NSB]);
      if (end) {  // hand the segment's (m, l of this half) to the epilogue warpgroup
        const int par = gseg & 1;
        if (!mbar_wait_warp(&c->seg_empty[par], ((gseg >> 1) & 1) ^ 1, &c->abort, p.err)) { ok = false; break; }
        if (active) {
          float s0 = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
          float s1 = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
          s0 += __shfl_xor_sync(0xffffffffu, s0, 2);
          s1 += __shfl_xor_sync(0xffffffffu, s1, 2);
          if ((ln & 3) == 0) {
            seg_ml[(par * R::SPLIT + part) * kBM + r0] = make_float2(m0, s0);
            seg_ml[(par * R::SPLIT + part) * kBM + r1] = make_float2(m1, s1);
          }
        }
        mbar_arrive(&c->seg_full[par]);
        ++gseg;
      }
      if (u + 1 < f.n) seg_next(sg, p.offsets, p.B);
    }
    if (!ok) break;
    g += f.n;
  }
}

// Epilogue of each finished segment: O / l in bf16 and the natural-log LSE
// for a whole sequence; for a piece of a split sequence, O / l in fp32 and
// the base-2 LSE m + log2(l) as a partial, in slot 0 (the piece starts
// inside the sequence) or 1 (it starts at the sequence's first tile) of the
// item.
template <int D, bool SPREAD>
__device__ void epilogue_role(const FwdParams& p, uint8_t* smem, FsCtl* c, uint32_t tbase) {
  using C = FsCfg<D>;
  using R = FsRoles<D>;
  const int r = threadIdx.x - R::kSoftmax;  // tile row == TMEM lane
  // the query of this row (spread layout: row 32 k + i holds query 16 k + i, i < 16)
  const int qr = SPREAD ? 16 * (r >> 5) + (r & 31) : r;
  const bool qrow_valid = (SPREAD ? (r & 31) < 16 : true) && qr < p.Lq;
  const uint32_t lane_base = static_cast<uint32_t>((r >> 5) * 32) << 16;
  const float2* seg_ml = reinterpret_cast<const float2*>(smem + C::kSeg);
  uint32_t gseg = 0;
  bool ok = true;
  for (uint32_t n = 0; ok; ++n) {
    FsDec f;
    if (!next_item(c, n, &f, &ok, p.err)) break;
    if (f.n == 0) continue;
    Seg sg;
    seg_load(sg, p.offsets, p.B, f.b, f.j);
    int seg_j0 = f.j;  // first tile of the current segment
    for (int u = 0; u < f.n && ok; ++u) {
      if (u > 0 && sg.j == 0) seg_j0 = 0;
      const bool end = u == f.n - 1 || sg.j == sg.nts - 1;
      if (end) {
        const int par = gseg & 1;
        const uint32_t ph = (gseg >> 1) & 1;
        if (!mbar_wait_warp(&c->seg_full[par], ph, &c->abort, p.err)) { ok = false; break; }
        const float m = seg_ml[(par * R::SPLIT) * kBM + r].x;
        float l = 0.f;
#pragma unroll
        for (int q = 0; q < R::SPLIT; ++q) l += seg_ml[(par * R::SPLIT + q) * kBM + r].y;
        mbar_arrive(&c->seg_empty[par]);
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        const bool whole = seg_j0 == 0 && sg.j == sg.nts - 1;
        const bool store = qrow_valid;
        const int slot = seg_j0 > 0 ? 0 : 1;
        const long long prow = (static_cast<long long>(f.slot) * 2 + slot) * kBM + qr;
        if (!mbar_wait_warp(&c->o_done[par], ph, &c->abort, p.err)) { ok = false; break; }
        tc_fence_after();
        // 32 columns at a time out of TMEM: a whole sequence keeps bf16
        // pairs until O is released; a piece is stored in fp32 at once.
        uint32_t w[D / 2];
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t o[32];
          tmem_ld32(tbase + lane_base + C::colO(par) + ch * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * inv_l);
          if (whole) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              w[16 * ch + i] = pack_bf16x2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1]));
          } else if (store) {
#pragma unroll
            for (int q = 0; q < 4; ++q) st_global_v8(p.part_o + prow * D + 32 * ch + 8 * q, o + 8 * q);
          }
        }
        tc_fence_before();
        mbar_arrive(&c->o_free[par]);
        ++gseg;
        if (store) {
          if (whole) {
            __nv_bfloat16* orow = p.out + ((static_cast<long long>(sg.b) * p.Lq + qr) * p.H + f.h) * D;
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) st_global_64B(orow + ch * 32, w + 16 * ch);
            p.lse[(static_cast<long long>(sg.b) * p.H + f.h) * p.Lq + qr] =
                l > 0.f ? (m + lg2_approx(l)) * kLn2 : -INFINITY;
          } else {
            p.part_lse[prow] = l > 0.f ? m + lg2_approx(l) : -INFINITY;
          }
        }
      }
      if (u + 1 < f.n) seg_next(sg, p.offsets, p.B);
    }
  }
}

template <int D, bool SPREAD>
__global__ void __launch_bounds__(FsRoles<D>::kThreads, 1)
    fwd_bs_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, const FwdParams p) {
  using C = FsCfg<D>;
  using R = FsRoles<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  FsCtl* c = reinterpret_cast<FsCtl*>(smem + C::kCtl);
  const int warp = warp_id(), lane = lane_id();
  if ((smem_addr(smem) & 1023) != 0) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrSmemAlign);
    return;
  }
  if (threadIdx.x == 0) {
    mbar_init(&c->q_full, 1);
    mbar_init(&c->q_empty, 1);
    for (int i = 0; i < C::NSK; ++i) {
      mbar_init(&c->k_full[i], 1);
      mbar_init(&c->k_empty[i], 1);
    }
    for (int i = 0; i < C::NSV; ++i) {
      mbar_init(&c->v_full[i], 1);
      mbar_init(&c->v_empty[i], 1);
    }
    for (int i = 0; i < 3; ++i) {
      mbar_init(&c->s_full[i], 1);
      mbar_init(&c->p_full[i], R::kSoftmax);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c->o_ready[i], 1);
      mbar_init(&c->o_done[i], 1);
      mbar_init(&c->o_free[i], kBM);
      mbar_init(&c->seg_full[i], R::kSoftmax);
      mbar_init(&c->seg_empty[i], kBM);
      mbar_init(&c->xbar[i], R::kSoftmax);
      mbar_init(&c->item_full[i], 1);
      mbar_init(&c->item_empty[i], R::kEpiWarp + 5);  // softmax + epilogue warps + the MMA warp
    }
    mbar_init(&c->drain, 1);
    c->abort = 0;
    fence_barrier_init();
  }
  if (warp == R::kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tq);
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
  }
  if (warp == R::kMmaWarp) {
    tmem_alloc(&c->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = c->tmem_base;
  if (warp < R::kEpiWarp) {
    if (SPREAD)
      softmax_spread<D>(p, smem, c, tbase);
    else
      softmax_role<D>(p, smem, c, tbase);
  } else if (warp < R::kEpiWarp + 4) {
    epilogue_role<D, SPREAD>(p, smem, c, tbase);
  } else if (warp == R::kProducerWarp) {
    if (lane == 0) producer_role<D, SPREAD>(&tq, &tk, &tv, p, smem, c);
  } else {
    mma_role<D>(p, smem, c, tbase);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == R::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// Merge of the pieces of split sequences, and the outputs of empty ones.
// One block per chunk boundary (item (c, h), c >= 1): the item starts inside
// sequence b (tile j > 0) when the boundary cuts b, and the block of b's
// first such boundary merges it: its first piece is in slot 1 of item
// (c - 1, h), the others in slot 0 of items (c .. c1, h), where c1 is the
// last consecutive item that starts inside b.  Threads take (query row, 8
// head-dim columns): O = sum_i 2^(lse_i - lse) O_i with lse = log2 sum_i
// 2^lse_i.  Every thread of the grid then checks one (sequence, head) and
// writes O = 0, LSE = -inf when the sequence is empty.
constexpr int kCombineThreads = 256;
template <int D>
__global__ void __launch_bounds__(kCombineThreads) fwd_combine_kernel(const FwdParams p) {
  const WorkHeader* hdr = p.hdr;
  if (!hdr->valid) return;
  const int nc = hdr->n_chunks;
  const long long idx = blockIdx.x + static_cast<long long>(p.H);  // items of chunks 1..
  if (idx < static_cast<long long>(nc) * p.H) {
    const int h = static_cast<int>(idx % p.H), c = static_cast<int>(idx / p.H);
    const QbItem it = p.qb_items[idx];
    const QbItem prev = p.qb_items[idx - p.H];
    // cut here, and by no earlier boundary
    if (it.j > 0 && !(prev.b == it.b && prev.j > 0)) {
      const int b = it.b, c0 = c - 1;
      int c1 = c;
      while (c1 + 1 < nc) {
        const QbItem nx = p.qb_items[static_cast<long long>(c1 + 1) * p.H + h];
        if (nx.b != b || nx.j == 0) break;
        ++c1;
      }
      constexpr int kGroups = D / 8;
      for (int w = threadIdx.x; w < p.Lq * kGroups; w += kCombineThreads) {
        const int r = w / kGroups, d0 = 8 * (w % kGroups);
        float lmax = -INFINITY;
        for (int cc = c0; cc <= c1; ++cc)
          lmax = fmaxf(lmax, p.part_lse[((static_cast<long long>(cc) * p.H + h) * 2 + (cc == c0)) * kBM + r]);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        float sw = 0.f;
        for (int cc = c0; cc <= c1; ++cc) {
          const long long prow = ((static_cast<long long>(cc) * p.H + h) * 2 + (cc == c0)) * kBM + r;
          const float wgt = ex2_approx(p.part_lse[prow] - lmax);
          sw += wgt;
          const float4* src = reinterpret_cast<const float4*>(p.part_o + prow * D + d0);
          const float4 v0 = src[0], v1 = src[1];
          acc[0] += wgt * v0.x;
          acc[1] += wgt * v0.y;
          acc[2] += wgt * v0.z;
          acc[3] += wgt * v0.w;
          acc[4] += wgt * v1.x;
          acc[5] += wgt * v1.y;
          acc[6] += wgt * v1.z;
          acc[7] += wgt * v1.w;
        }
        const float inv = 1.f / sw;
        __nv_bfloat16* orow = p.out + ((static_cast<long long>(b) * p.Lq + r) * p.H + h) * D + d0;
        *reinterpret_cast<uint4*>(orow) =
            make_uint4(pack_bf16x2(acc[0] * inv, acc[1] * inv), pack_bf16x2(acc[2] * inv, acc[3] * inv),
                       pack_bf16x2(acc[4] * inv, acc[5] * inv), pack_bf16x2(acc[6] * inv, acc[7] * inv));
        if (d0 == 0) p.lse[(static_cast<long long>(b) * p.H + h) * p.Lq + r] = (lmax + lg2_approx(sw)) * kLn2;
      }
    }
  }
  // empty sequences
  const long long nbh = static_cast<long long>(p.B) * p.H;
  const long long nthreads = static_cast<long long>(gridDim.x) * kCombineThreads;
  for (long long i = static_cast<long long>(blockIdx.x) * kCombineThreads + threadIdx.x; i < nbh;
       i += nthreads) {
    const int h = static_cast<int>(i % p.H), b = static_cast<int>(i / p.H);
    if (p.offsets[b + 1] != p.offsets[b]) continue;
    float* lrow = p.lse + (static_cast<long long>(b) * p.H + h) * p.Lq;
    for (int r = 0; r < p.Lq; ++r) {
      __nv_bfloat16* orow = p.out + ((static_cast<long long>(b) * p.Lq + r) * p.H + h) * D;
      for (int d = 0; d < D; d += 8) *reinterpret_cast<uint4*>(orow + d) = make_uint4(0, 0, 0, 0);
      lrow[r] = -INFINITY;
    }
  }
}

template <int D, bool SPREAD>
cudaError_t launch_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     const FwdParams& p, int grid, cudaStream_t s) {
  using C = FsCfg<D>;
  static_assert(C::kSmem <= 232448, "shared memory budget");
  static_assert(sizeof(FsCtl) <= 512, "control block");
  static_assert(C::NSK <= 4 && C::NSV <= 4, "ring depth");
  auto kern = fwd_bs_kernel<D, SPREAD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  kern<<<grid, FsRoles<D>::kThreads, C::kSmem, s>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

bool fwd_bs_supported(int Lq) { return Lq >= 1 && Lq <= kBM; }
bool fwd_bs_spread(int Lq) { return Lq >= 1 && Lq <= 64; }

cudaError_t launch_fwd_bs(int D, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const FwdParams& p, int grid, cudaStream_t s) {
  if (!fwd_bs_supported(p.Lq)) return cudaErrorInvalidValue;
  if (fwd_bs_spread(p.Lq)) {
    if (D == 128) return launch_t<128, true>(tq, tk, tv, p, grid, s);
    return launch_t<64, true>(tq, tk, tv, p, grid, s);
  }
  if (D == 128) return launch_t<128, false>(tq, tk, tv, p, grid, s);
  return launch_t<64, false>(tq, tk, tv, p, grid, s);
}

cudaError_t launch_fwd_combine(int D, const FwdParams& p, int sms, cudaStream_t s) {
  // one block per chunk boundary (the chunk list holds at most chunk_cap =
  // ceil(2 * sms / H) chunks per head), and at least one thread per
  // (sequence, head) for the empty-sequence pass
  const long long boundaries = std::max<long long>(1, ((2LL * sms + p.H - 1) / p.H) * p.H);
  const long long for_empty = (static_cast<long long>(p.B) * p.H + kCombineThreads - 1) / kCombineThreads;
  const int grid = static_cast<int>(std::max(boundaries, std::min<long long>(for_empty, 4LL * sms)));
  if (D == 128)
    fwd_combine_kernel<128><<<grid, kCombineThreads, 0, s>>>(p);
  else
    fwd_combine_kernel<64><<<grid, kCombineThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace jfa
