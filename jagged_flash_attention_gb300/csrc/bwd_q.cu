// Self-attention backward, pass 2 of 2: dQ for sm_103a.
//
// The dQ part of the five backward products ("Optimizing Jagged Flash
// Attention with TLX", "2-CTA collaborative MMA") computed query-outer like
// the forward, so that dQ of a query tile accumulates in tensor memory over
// all of its key tiles and is written once, in bf16, with no cross-CTA
// reduction (the fp32 reduce-add the page stages for broadcast-Q, section
// "Multi-stage dQ staging", has no counterpart here).  Per key tile j:
//   S_j  = Q K_j^T      (SS, K-major / K-major) -> TMEM S[j%2]
//   dP_j = dO V_j^T     (SS)                    -> TMEM dP
//   P = exp2(S * scale*log2e - LSE*log2e), dS = P (dP - Delta)   (fp32)
//   dS (bf16) over S[j%2]'s columns; dQ += dS K_j  (TS, B = K MN-major)
// Issue order: dQ(j-1), dP(j), S(j+1), so S(j+1) runs while the math warps
// turn S(j), dP(j) into dS(j).
//
// CTA = 10 warps: warps 0-7 math (warp w: query row 32*(w%4)+lane, key
// columns 64*(w/4)..) and the dQ epilogue, warp 8 TMA producer, warp 9 MMA.
#include "common.cuh"
#include "ptx.cuh"

namespace jfa {
namespace {

constexpr int kThreads = 320;
constexpr int kMath = 256;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct QCfg {
  static constexpr int NSK = (D == 128) ? 3 : 4;  // K ring depth
  static constexpr int NSV = (D == 128) ? 2 : 4;  // V ring depth
  static constexpr int kTile = kBM * D * 2;
  static constexpr int kSlabs = D / 64;
  static constexpr int kQ = 0;
  static constexpr int kDO = kTile;
  static constexpr int kK = 2 * kTile;
  static constexpr int kV = kK + NSK * kTile;
  static constexpr int kCtl = kV + NSV * kTile;
  static constexpr int kSmem = kCtl + 512;
  __host__ __device__ static constexpr uint32_t colS(uint32_t b) { return 128u * b; }
  static constexpr uint32_t kColDP = 256, kColDQ = 384;
};

struct QCtl {
  uint64_t qdo_full, qdo_empty;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t sd_full, ds_full;
  uint64_t dq_full, dq_free;
  uint64_t item_full[2], item_empty[2];
  uint64_t drain;
  int item_slot[2];
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ int cdiv(int a, int b) { return (a + b - 1) / b; }

struct QItem {
  int b, h, t;
  int off0, L;
  int q_lo, nq, shift, row;  // query tile: first local row, valid rows, box shift, TMA row
  int n_kv;
};

template <bool CAUSAL>
__device__ __forceinline__ QItem decode(const BwdParams& p, int idx, int T) {
  QItem f;
  const Item it = p.items[idx];
  f.b = it.x;
  f.h = it.y >> 16;
  f.t = it.y & 0xffff;
  f.off0 = p.offsets[f.b];
  f.L = p.offsets[f.b + 1] - f.off0;
  f.q_lo = f.t * kBM;
  f.nq = min(kBM, f.L - f.q_lo);
  const int start = f.off0 + f.q_lo;
  f.shift = max(0, start + kBM - T);
  f.row = start - f.shift;
  f.n_kv = CAUSAL ? cdiv(f.q_lo + f.nq, kBN) : cdiv(f.L, kBN);
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
    mbar_arrive_expect_tx(&c->qdo_full, 2 * C::kTile);
#pragma unroll
    for (int s = 0; s < C::kSlabs; ++s) {
      tma_load_3d(smem + C::kQ + s * 16384, tq, &c->qdo_full, s * 64, f.h, f.row);
      tma_load_3d(smem + C::kDO + s * 16384, tdo, &c->qdo_full, s * 64, f.h, f.row);
    }
    ++it;
    for (int j = 0; j < f.n_kv; ++j) {
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
  uint32_t it = 0, nk = 0, nv = 0, g = 0;  // g: key tiles processed over all items
  bool ok = true, issued = false;
  // Descriptors built once; per tile and K step only adds remain.
  const uint64_t dq_k = smem_desc_sw128(smem_addr(smem + C::kQ), 16, 1024);
  const uint64_t ddo_k = smem_desc_sw128(smem_addr(smem + C::kDO), 16, 1024);
  const uint64_t dk_k0 = smem_desc_sw128(smem_addr(smem + C::kK), 16, 1024);
  const uint64_t dk_m0 = smem_desc_sw128(smem_addr(smem + C::kK), 16384, 1024);
  const uint64_t dv_k0 = smem_desc_sw128(smem_addr(smem + C::kV), 16, 1024);
  auto issue_s = [&](uint32_t buf, uint32_t kidx) {
    const uint64_t dk = desc_add(dk_k0, (kidx % C::NSK) * C::kTile);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
      mma_ss(tbase + C::colS(buf), desc_add(dq_k, off), desc_add(dk, off), id_s, k > 0);
    }
  };
  auto issue_dp = [&](uint32_t vidx) {
    const uint64_t dv = desc_add(dv_k0, (vidx % C::NSV) * C::kTile);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
      mma_ss(tbase + C::kColDP, desc_add(ddo_k, off), desc_add(dv, off), id_s, k > 0);
    }
  };
  auto issue_dq = [&](uint32_t buf, uint32_t kidx, bool acc) {
    // A = dS (bf16 in S[buf]): keys 0-63 packed at +0, keys 64-127 at +64.
    const uint64_t dk = desc_add(dk_m0, (kidx % C::NSK) * C::kTile);
#pragma unroll
    for (int k = 0; k < kBN / 16; ++k) {
      const uint32_t acol = k * 8 + (k >= 4 ? 32 : 0);
      mma_ts(tbase + C::kColDQ, tbase + C::colS(buf) + acol, desc_add(dk, k * 2048), id_dq,
             acc || (k > 0));
    }
  };
  for (uint32_t n = 0; ok; ++n) {
    const int idx = next_item(c, n, false, &ok, p.err);
    if (idx < 0) break;
    const QItem f = decode<CAUSAL>(p, idx, T);
    if (!mbar_wait(&c->qdo_full, it & 1, &c->abort, p.err)) break;
    const uint32_t k0 = nk, g0 = g;  // K tile index and global tile index of j = 0
    // S(0)
    if (!mbar_wait(&c->k_full[k0 % C::NSK], (k0 / C::NSK) & 1, &c->abort, p.err)) break;
    tc_fence_after();
    issue_s(g0 & 1, k0);
    issued = true;
    for (int j = 0; j < f.n_kv && ok; ++j) {
      const uint32_t gj = g0 + j;
      if (!mbar_wait(&c->v_full[nv % C::NSV], (nv / C::NSV) & 1, &c->abort, p.err)) { ok = false; break; }
      if (j > 0) {  // dQ += dS(j-1) K(j-1): frees the dP buffer's reader first
        if (!mbar_wait(&c->ds_full, (gj - 1) & 1, &c->abort, p.err)) { ok = false; break; }
        if (j == 1 && !mbar_wait(&c->dq_free, (it & 1) ^ 1, &c->abort, p.err)) { ok = false; break; }
        tc_fence_after();
        issue_dq((gj - 1) & 1, k0 + j - 1, j > 1);
        mma_commit(&c->k_empty[(k0 + j - 1) % C::NSK]);
      }
      issue_dp(nv);  // dP(j) = dO V(j)^T
      mma_commit(&c->sd_full);  // S(j) and dP(j) ready
      mma_commit(&c->v_empty[nv % C::NSV]);
      ++nv;
      if (j + 1 < f.n_kv) {  // S(j+1) into the other buffer (its dS(j-1) is consumed)
        const uint32_t kk = k0 + j + 1;
        if (!mbar_wait(&c->k_full[kk % C::NSK], (kk / C::NSK) & 1, &c->abort, p.err)) { ok = false; break; }
        issue_s((gj + 1) & 1, kk);
      }
    }
    if (!ok) break;
    const uint32_t gl = g0 + f.n_kv - 1;
    if (!mbar_wait(&c->ds_full, gl & 1, &c->abort, p.err)) break;
    if (f.n_kv == 1 && !mbar_wait(&c->dq_free, (it & 1) ^ 1, &c->abort, p.err)) break;
    tc_fence_after();
    issue_dq(gl & 1, k0 + f.n_kv - 1, f.n_kv > 1);
    mma_commit(&c->k_empty[(k0 + f.n_kv - 1) % C::NSK]);
    mma_commit(&c->dq_full);
    mma_commit(&c->qdo_empty);
    nk += f.n_kv;
    g += f.n_kv;
    ++it;
  }
  if (issued) {
    mma_commit(&c->drain);
    drain_wait(&c->drain, 0, p.err);
  }
}

template <int D, bool CAUSAL>
__device__ void math_role(const BwdParams& p, QCtl* c, uint32_t tbase) {
  using C = QCfg<D>;
  const int r = threadIdx.x & 127;    // query row of the tile == TMEM lane
  const int half = threadIdx.x >> 7;  // key columns [64*half, 64*half + 64)
  const uint32_t lane_base = static_cast<uint32_t>((r >> 5) * 32) << 16;
  const int T = p.hdr->T;
  const float sl2 = p.scale_log2;
  uint32_t it = 0, g = 0;
  bool ok = true;
  for (uint32_t n = 0; ok; ++n) {
    const int idx = next_item(c, n, true, &ok, p.err);
    if (idx < 0) break;
    const QItem f = decode<CAUSAL>(p, idx, T);
    const int qi = f.q_lo - f.shift + r;  // local query index of this row
    const bool row_valid = r >= f.shift && r < f.shift + f.nq;
    float lse2 = INFINITY, dlt = 0.f;  // rows outside the sequence: P = 0
    if (row_valid) {
      const long long si = static_cast<long long>(f.h) * T + f.off0 + qi;
      lse2 = p.lse[si] * kLog2e;
      dlt = p.delta[si];
    }
    for (int j = 0; j < f.n_kv; ++j, ++g) {
      if (!mbar_wait_warp(&c->sd_full, g & 1, &c->abort, p.err)) { ok = false; break; }
      tc_fence_after();
      const uint32_t ts = tbase + lane_base + C::colS(g & 1);
      const KvTile kt = kv_tile(f.off0, f.L, j, T);
      const int key0 = j * kBN - kt.shift;  // local key index of column 0
      const bool need_mask =
          kt.nk < kBN || kt.shift > 0 || (CAUSAL && key0 + kBN - 1 > f.q_lo - f.shift);
      const int c_lo = kt.shift, c_hi = kt.shift + kt.nk;
      const int c_causal = qi - key0;  // last admissible column when causal
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const int cbase = 64 * half + 32 * ch;
        uint32_t sraw[32], praw[32];
        tmem_ld32(ts + cbase, sraw);
        tmem_ld32(tbase + lane_base + C::kColDP + cbase, praw);
        tmem_wait_ld();
        uint32_t dk[16];
#pragma unroll
        for (int cc = 0; cc < 32; cc += 2) {
          const int col = cbase + cc;
          float p0 = ex2_approx(fmaf(__uint_as_float(sraw[cc]), sl2, -lse2));
          float p1 = ex2_approx(fmaf(__uint_as_float(sraw[cc + 1]), sl2, -lse2));
          if (need_mask) {
            const bool k0 = col >= c_lo && col < c_hi && (!CAUSAL || col <= c_causal);
            const bool k1 = col + 1 >= c_lo && col + 1 < c_hi && (!CAUSAL || col + 1 <= c_causal);
            p0 = k0 ? p0 : 0.f;
            p1 = k1 ? p1 : 0.f;
          }
          const float d0 = p0 * (__uint_as_float(praw[cc]) - dlt);
          const float d1 = p1 * (__uint_as_float(praw[cc + 1]) - dlt);
          dk[cc / 2] = pack_bf16x2(d0, d1);
        }
        // Packed dS of key columns cbase.. at cbase / 2 + 32 * half: inside
        // the fp32 columns this half has already read.
        tmem_st16(ts + cbase / 2 + 32 * half, dk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&c->ds_full);
    }
    if (!ok) break;
    // Epilogue: dQ = scale * acc in bf16 (this warp's half of the head dim).
    if (!mbar_wait_warp(&c->dq_full, it & 1, &c->abort, p.err)) break;
    tc_fence_after();
    __nv_bfloat16* dst = p.dq + ((static_cast<long long>(f.off0) + qi) * p.H + f.h) * D;
#pragma unroll
    for (int ch = 0; ch < D / 64; ++ch) {
      const int dbase = (D / 2) * half + 32 * ch;
      uint32_t v[32];
      tmem_ld32(tbase + lane_base + C::kColDQ + dbase, v);
      tmem_wait_ld();
      uint32_t w[16];
#pragma unroll
      for (int i2 = 0; i2 < 16; ++i2)
        w[i2] = pack_bf16x2(__uint_as_float(v[2 * i2]) * p.scale,
                            __uint_as_float(v[2 * i2 + 1]) * p.scale);
      if (row_valid) {
        uint4* d4 = reinterpret_cast<uint4*>(dst + dbase);
        d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
        d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
        d4[2] = make_uint4(w[8], w[9], w[10], w[11]);
        d4[3] = make_uint4(w[12], w[13], w[14], w[15]);
      }
    }
    tc_fence_before();
    mbar_arrive(&c->dq_free);
    ++it;
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
    mbar_init(&c->sd_full, 1);
    mbar_init(&c->ds_full, kMath);
    mbar_init(&c->dq_full, 1);
    mbar_init(&c->dq_free, kMath);
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
