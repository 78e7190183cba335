// Jagged flash attention forward for sm_103a.
//
// Method: "Optimizing Jagged Flash Attention with TLX" (pytorch.org),
// section 2.1 (role-specialised warps, hand-allocated SMEM/TMEM buffers with
// S and P sharing one TMEM allocation while the PV accumulator keeps its
// own, persistent CTAs) and section 2.2 (longest-first scheduling, masking
// only the ragged tail tile); per-row math from "cuTile Kernels - FMHA
// Implementation", "Flash Attention Algorithm" and "exp2 + flush_to_zero"
// (online softmax in base 2 with the scale folded into one multiply).
//
// CTA = 6 warps, one CTA per SM, looping over work items (b, h, q-tile):
//   warps 0-3  softmax / correction / epilogue; thread r owns query row r
//              (TMEM lane r) of the 128-row tile
//   warp 4     TMA producer (Q once per item, K and V tiles into NS-deep
//              rings) and the dynamic work ticket
//   warp 5     TMEM allocation and the single-thread tcgen05 MMA issuer
// TMEM (512 columns): S0 [0,128), S1 [128,256), O [256, 256+D).  P (bf16)
// overwrites the first 64 columns of the S buffer it was computed from and
// is read from TMEM by the PV MMA.
#include "common.cuh"
#include "ptx.cuh"

namespace jfa {
namespace {

constexpr int kFwdThreads = 192;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct FwdCfg {
  static constexpr int NS = (D == 128) ? 2 : 4;  // K and V ring depth
  static constexpr int kTile = kBM * D * 2;      // bytes of a 128-row bf16 tile
  static constexpr int kSlabs = D / 64;          // 64-column (128 B) slabs per row
  static constexpr int kQ = 0;
  static constexpr int kK = kTile;
  static constexpr int kV = kK + NS * kTile;
  static constexpr int kCtl = kV + NS * kTile;  // barriers and small state
  static constexpr int kSmem = kCtl + 512;
  static constexpr uint32_t kColO = 256;
};

struct FwdCtl {
  uint64_t q_full, q_empty;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], p_full[2];
  uint64_t o_ready, o_free;
  uint64_t item_full[2], item_empty[2];
  uint64_t drain;
  int item_slot[2];
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

struct FwdTile {
  int b, h, t;
  int off0, L;
  int q_lo;     // local index of the tile's first query row
  int nq;       // valid query rows
  int q_shift;  // rows the Q box was moved back to stay inside [0, T)
  int q_row;    // TMA row coordinate of the Q box
  int n_kv;     // key tiles to visit
};

template <bool BCAST, bool CAUSAL>
__device__ __forceinline__ FwdTile decode(const FwdParams& p, int idx, int T) {
  FwdTile f;
  const Item it = p.items[idx];
  f.b = it.x;
  f.h = it.y >> 16;
  f.t = it.y & 0xffff;
  f.off0 = p.offsets[f.b];
  f.L = p.offsets[f.b + 1] - f.off0;
  f.q_lo = f.t * kBM;
  if (BCAST) {
    f.nq = min(kBM, p.Lq - f.q_lo);
    f.q_shift = 0;
    f.q_row = f.q_lo;
    f.n_kv = cdiv(f.L, kBN);
  } else {
    f.nq = min(kBM, f.L - f.q_lo);
    const int start = f.off0 + f.q_lo;
    f.q_shift = max(0, start + kBM - T);
    f.q_row = start - f.q_shift;
    f.n_kv = CAUSAL ? cdiv(f.q_lo + f.nq, kBN) : cdiv(f.L, kBN);
  }
  return f;
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

// Item queue consumer: returns the item index or -1 at the end.  `warp`:
// called by a whole warp (lane 0 arrives) rather than by a single thread.
__device__ __forceinline__ int next_item(FwdCtl* c, uint32_t n, bool warp, bool* ok, int* err) {
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
                              const FwdParams& p, uint8_t* smem, FwdCtl* c) {
  using C = FwdCfg<D>;
  const int n_items = p.hdr->n_items;
  const int T = p.hdr->T;
  uint32_t it = 0, kv = 0, nk_issued = 0, nv_issued = 0;
  bool ok = true;
  for (uint32_t n = 0; ok; ++n) {
    const int slot = n & 1;
    if (!mbar_wait(&c->item_empty[slot], ((n >> 1) & 1) ^ 1, &c->abort, p.err)) break;
    const int idx = atomicAdd(&p.hdr->ticket, 1);
    c->item_slot[slot] = idx < n_items ? idx : -1;
    mbar_arrive(&c->item_full[slot]);
    if (idx >= n_items) break;
    const FwdTile f = decode<BCAST, CAUSAL>(p, idx, T);
    if (f.n_kv == 0) continue;
    if (!mbar_wait(&c->q_empty, (it & 1) ^ 1, &c->abort, p.err)) break;
    mbar_arrive_expect_tx(&c->q_full, C::kTile);
#pragma unroll
    for (int s = 0; s < C::kSlabs; ++s)
      tma_load_3d(smem + C::kQ + s * 16384, tq, &c->q_full, s * 64, f.h, f.q_row);
    ++it;
    for (int j = 0; j < f.n_kv; ++j, ++kv) {
      const int st = kv % C::NS;
      const uint32_t ph = ((kv / C::NS) & 1) ^ 1;
      const KvTile kt = kv_tile(f.off0, f.L, j, T);
      if (!mbar_wait(&c->k_empty[st], ph, &c->abort, p.err)) { ok = false; break; }
      mbar_arrive_expect_tx(&c->k_full[st], C::kTile);
#pragma unroll
      for (int s = 0; s < C::kSlabs; ++s)
        tma_load_3d(smem + C::kK + st * C::kTile + s * 16384, tk, &c->k_full[st], s * 64, f.h,
                    kt.row);
      ++nk_issued;
      if (!mbar_wait(&c->v_empty[st], ph, &c->abort, p.err)) { ok = false; break; }
      mbar_arrive_expect_tx(&c->v_full[st], C::kTile);
#pragma unroll
      for (int s = 0; s < C::kSlabs; ++s)
        tma_load_3d(smem + C::kV + st * C::kTile + s * 16384, tv, &c->v_full[st], s * 64, f.h,
                    kt.row);
      ++nv_issued;
    }
  }
  // Drain: make sure every copy this CTA issued has landed before exit.
  if (it > 0) drain_wait(&c->q_full, (it - 1) & 1, p.err);
  for (uint32_t g = nk_issued > C::NS ? nk_issued - C::NS : 0; g < nk_issued; ++g)
    drain_wait(&c->k_full[g % C::NS], (g / C::NS) & 1, p.err);
  for (uint32_t g = nv_issued > C::NS ? nv_issued - C::NS : 0; g < nv_issued; ++g)
    drain_wait(&c->v_full[g % C::NS], (g / C::NS) & 1, p.err);
}

template <int D, bool CAUSAL, bool BCAST>
__device__ void mma_role(const FwdParams& p, uint8_t* smem, FwdCtl* c, uint32_t tbase) {
  using C = FwdCfg<D>;
  const int T = p.hdr->T;
  const uint32_t id_s = idesc_bf16_f32(kBM, kBN, false, false);
  const uint32_t id_pv = idesc_bf16_f32(kBM, D, false, true);
  const uint32_t sq = smem_addr(smem + C::kQ);
  uint32_t it = 0, kv = 0;
  // PV completions observed so far through o_ready.  A parity wait is only
  // valid while the barrier is at most one phase ahead of the waiter, so PV_x
  // is issued only after PV_{x-1} has been observed (free in steady state:
  // the softmax warps waited for PV_{x-1} before releasing P_x).
  uint32_t pv_seen = 0;
  auto wait_pv = [&](uint32_t x) -> bool {
    if (x < pv_seen) return true;
    if (!mbar_wait(&c->o_ready, x & 1, &c->abort, p.err)) return false;
    pv_seen = x + 1;
    return true;
  };
  bool ok = true;
  bool issued = false;
  for (uint32_t n = 0; ok; ++n) {
    const int idx = next_item(c, n, false, &ok, p.err);
    if (idx < 0) break;
    const FwdTile f = decode<BCAST, CAUSAL>(p, idx, T);
    if (f.n_kv == 0) continue;
    if (!mbar_wait(&c->q_full, it & 1, &c->abort, p.err)) break;
    for (int j = 0; j <= f.n_kv && ok; ++j) {
      if (j < f.n_kv) {
        const uint32_t g = kv + j;
        const int st = g % C::NS;
        const uint32_t buf = g & 1;
        if (!mbar_wait(&c->k_full[st], (g / C::NS) & 1, &c->abort, p.err)) { ok = false; break; }
        // S buffer `buf` last held P_{g-2}; its PV must have finished reading it.
        if (g >= 2 && !wait_pv(g - 2)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sk = smem_addr(smem + C::kK + st * C::kTile);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
          mma_ss(tmem_at(tbase, 0, buf * 128), smem_desc_sw128(sq + off, 16, 1024),
                 smem_desc_sw128(sk + off, 16, 1024), id_s, k > 0);
        }
        mma_commit(&c->s_full[buf]);
        mma_commit(&c->k_empty[st]);
        if (j == f.n_kv - 1) mma_commit(&c->q_empty);
        issued = true;
      }
      if (j >= 1) {
        const uint32_t g = kv + j - 1;
        const int st = g % C::NS;
        const uint32_t buf = g & 1;
        if (!mbar_wait(&c->p_full[buf], (g >> 1) & 1, &c->abort, p.err)) { ok = false; break; }
        if (!mbar_wait(&c->v_full[st], (g / C::NS) & 1, &c->abort, p.err)) { ok = false; break; }
        if (j == 1 && !mbar_wait(&c->o_free, (it & 1) ^ 1, &c->abort, p.err)) { ok = false; break; }
        if (g >= 1 && !wait_pv(g - 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sv = smem_addr(smem + C::kV + st * C::kTile);
#pragma unroll
        for (int k = 0; k < kBN / 16; ++k) {
          mma_ts(tmem_at(tbase, 0, C::kColO), tmem_at(tbase, 0, buf * 128 + k * 8),
                 smem_desc_sw128(sv + k * 2048, 16384, 1024), id_pv, (j > 1) || (k > 0));
        }
        mma_commit(&c->v_empty[st]);
        mma_commit(&c->o_ready);
      }
    }
    kv += f.n_kv;
    ++it;
  }
  if (issued) {
    mma_commit(&c->drain);
    drain_wait(&c->drain, 0, p.err);
  }
}

template <int D, bool CAUSAL, bool BCAST>
__device__ void softmax_role(const FwdParams& p, FwdCtl* c, uint32_t tbase) {
  using C = FwdCfg<D>;
  const int r = threadIdx.x;  // row of the tile == TMEM lane
  const int warp = r >> 5;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  const int T = p.hdr->T;
  const float sl2 = p.scale_log2;
  uint32_t it = 0, kv = 0;
  bool ok = true;
  for (uint32_t n = 0; ok; ++n) {
    const int idx = next_item(c, n, true, &ok, p.err);
    if (idx < 0) break;
    const FwdTile f = decode<BCAST, CAUSAL>(p, idx, T);
    const int qi = f.q_lo - f.q_shift + r;  // local query index of this row
    const bool row_valid = r >= f.q_shift && r < f.q_shift + f.nq;
    __nv_bfloat16* orow;
    float* lrow;
    if (BCAST) {
      orow = p.out + ((static_cast<long long>(f.b) * p.Lq + qi) * p.H + f.h) * D;
      lrow = p.lse + (static_cast<long long>(f.b) * p.H + f.h) * p.Lq + qi;
    } else {
      orow = p.out + ((static_cast<long long>(f.off0) + qi) * p.H + f.h) * D;
      lrow = p.lse + static_cast<long long>(f.h) * T + f.off0 + qi;
    }
    if (f.n_kv == 0) {  // empty broadcast sequence: O = 0, LSE = -inf
      if (row_valid) {
        for (int d = 0; d < D; d += 8) *reinterpret_cast<uint4*>(orow + d) = make_uint4(0, 0, 0, 0);
        *lrow = -INFINITY;
      }
      continue;
    }
    float m_run = -INFINITY, l_run = 0.f;
    for (int j = 0; j < f.n_kv; ++j) {
      const uint32_t g = kv + j;
      const uint32_t buf = g & 1;
      if (!mbar_wait_warp(&c->s_full[buf], (g >> 1) & 1, &c->abort, p.err)) { ok = false; break; }
      tc_fence_after();
      const uint32_t ts = tbase + lane_base + buf * 128;
      uint32_t raw[4][32];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) tmem_ld32(ts + ch * 32, raw[ch]);
      tmem_wait_ld();
      float s[128];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch)
#pragma unroll
        for (int i = 0; i < 32; ++i) s[ch * 32 + i] = __uint_as_float(raw[ch][i]);
      const KvTile kt = kv_tile(f.off0, f.L, j, T);
      const int key0 = j * kBN - kt.shift;  // local key index of column 0
      const bool need_mask =
          kt.nk < kBN || kt.shift > 0 || (CAUSAL && key0 + kBN - 1 > f.q_lo - f.q_shift);
      if (need_mask) {
        // Peeled tail: only the ragged last tile (and the diagonal tile when
        // causal) pays for the per-element mask.
        const int c_lo = kt.shift, c_hi = kt.shift + kt.nk;
        const int c_causal = qi - key0;  // last admissible column when causal
#pragma unroll
        for (int cc = 0; cc < 128; ++cc) {
          const bool keep = cc >= c_lo && cc < c_hi && (!CAUSAL || cc <= c_causal);
          s[cc] = keep ? s[cc] : -INFINITY;
        }
      }
      float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
      for (int cc = 4; cc < 128; cc += 4) {
        mx0 = fmaxf(mx0, s[cc]);
        mx1 = fmaxf(mx1, s[cc + 1]);
        mx2 = fmaxf(mx2, s[cc + 2]);
        mx3 = fmaxf(mx3, s[cc + 3]);
      }
      const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
      const float m_new = fmaxf(m_run, mx * sl2);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2_approx(m_run - m_use);
      float sum0 = 0.f, sum1 = 0.f;
      uint32_t pk[4][16];
#pragma unroll
      for (int cc = 0; cc < 128; cc += 2) {
        const float p0 = ex2_approx(fmaf(s[cc], sl2, -m_use));
        const float p1 = ex2_approx(fmaf(s[cc + 1], sl2, -m_use));
        sum0 += p0;
        sum1 += p1;
        pk[cc / 32][(cc % 32) / 2] = pack_bf16x2(p0, p1);
      }
      l_run = l_run * alpha + (sum0 + sum1);
      m_run = m_new;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) tmem_st16(ts + ch * 16, pk[ch]);
      if (j > 0) {
        // Correction: rescale the running O once PV_{g-1} has landed.
        if (!mbar_wait_warp(&c->o_ready, (g - 1) & 1, &c->abort, p.err)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          const uint32_t to = tbase + lane_base + C::kColO;
#pragma unroll
          for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t o[32];
            tmem_ld32(to + ch * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(to + ch * 32, o);
          }
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&c->p_full[buf]);
    }
    if (!ok) break;
    kv += f.n_kv;
    // Epilogue: O / l in bf16 and the natural-log LSE.
    if (!mbar_wait_warp(&c->o_ready, (kv - 1) & 1, &c->abort, p.err)) break;
    tc_fence_after();
    const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
    const uint32_t to = tbase + lane_base + C::kColO;
#pragma unroll
    for (int ch = 0; ch < D / 32; ++ch) {
      uint32_t o[32];
      tmem_ld32(to + ch * 32, o);
      tmem_wait_ld();
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 16; ++i)
        w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
      if (row_valid) {
        uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        dst[2] = make_uint4(w[8], w[9], w[10], w[11]);
        dst[3] = make_uint4(w[12], w[13], w[14], w[15]);
      }
    }
    if (row_valid) *lrow = l_run > 0.f ? (m_run + lg2_approx(l_run)) * kLn2 : -INFINITY;
    tc_fence_before();
    mbar_arrive(&c->o_free);
    ++it;
  }
}

template <int D, bool CAUSAL, bool BCAST>
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
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(&c->k_full[i], 1);
      mbar_init(&c->k_empty[i], 1);
      mbar_init(&c->v_full[i], 1);
      mbar_init(&c->v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c->s_full[i], 1);
      mbar_init(&c->p_full[i], kBM);
      mbar_init(&c->item_full[i], 1);
      mbar_init(&c->item_empty[i], 5);  // 4 softmax warps + the MMA thread
    }
    mbar_init(&c->o_ready, 1);
    mbar_init(&c->o_free, kBM);
    mbar_init(&c->drain, 1);
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

  if (warp < 4) {
    softmax_role<D, CAUSAL, BCAST>(p, c, tbase);
  } else if (warp == kProducerWarp) {
    if (lane == 0) producer_role<D, CAUSAL, BCAST>(&tq, &tk, &tv, p, smem, c);
  } else {
    if (lane == 0) mma_role<D, CAUSAL, BCAST>(p, smem, c, tbase);
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
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const FwdParams& p, int grid, cudaStream_t s) {
  using C = FwdCfg<D>;
  static_assert(C::kSmem <= 232448, "shared memory budget");
  static_assert(sizeof(FwdCtl) <= 512, "control block");
  auto kern = fwd_kernel<D, CAUSAL, BCAST>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kFwdThreads, C::kSmem, s>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd(int D, bool causal, bool bcast, const CUtensorMap& tq, const CUtensorMap& tk,
                       const CUtensorMap& tv, const FwdParams& p, int grid, cudaStream_t s) {
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
