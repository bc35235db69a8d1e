// fwd.cu -- fused attention forward for sm_103a.
//
// One kernel computes O = softmax(scale Q K^T [+ causal mask]) V and the
// per-row logsumexp, keeping S and P on chip ("Gemini 3 Flash的注意力内核重写：
// 算子融合如何实现亚毫秒级推理", §1 内核融合策略: load Q/K/V blocks, do QK^T,
// softmax and PV on chip, write only O).  Keys are visited in tiles with a
// running max and running sum (same page, §3 在线softmax算法); tiles of keys
// wholly above the causal diagonal are never visited ("提示词再优也救不了的性能
// 黑洞…", 第一章, causal=True skips the upper triangle).
//
// GB300 mapping (one CTA per SM; 320 threads, 384 with bf16 inputs):
//   * the CTA owns two 128-row query tiles (256 rows) of one (batch, head),
//     one on grids small enough for one wave; they share one K/V stream;
//   * warp 8 issues TMA loads: both Q tiles once, then K_j and V_j into
//     STAGES-deep rings of 128-byte-swizzled shared-memory tiles;
//   * warp 9 (one thread) issues tcgen05 MMAs: S_t = Q_t K_j^T into TMEM
//     (fp32, 128 lanes x 128 columns per tile) and O_t += P_t V_j with P_t
//     read straight from TMEM;
//   * warps 0-3 and 4-7 are the softmax warpgroups of tile 0 and tile 1; a
//     thread owns one query row (= one TMEM lane).  Per key tile it reads its
//     128 scores, updates the running max, rescales the running sum and the
//     TMEM O row when the max has grown by more than 2^8 (the reference max
//     is otherwise kept; the final normalisation by the same reference makes
//     the result identical), writes P = 2^(s*scale*log2e - m) as f16 into
//     TMEM (over the S columns at d = 128, in columns of its own at d = 64),
//     and hands the tile back to the MMA warp.  While one
//     warpgroup does its softmax the tensor core works on the other tile.
//   * P V runs in f16 whatever the input type: P rounded to f16 (11
//     significant bits) errs 8x less than bf16 (8 bits), which keeps O within
//     its error bound on rows dominated by a few keys.  The MMA takes both
//     operands in one type, so for bf16 inputs warps 10-11 convert each V
//     tile to f16 in shared memory, in place, between its TMA landing and its
//     first P V (exact for 2^-14 <= |v| <= 65504 and for 0; smaller
//     magnitudes are carried with an absolute error below 2^-25).
//   * epilogue: O_t / l rounded to the input type (and, when asked for, an
//     fp32 copy of the same quotient), lse = (m + log2 l) ln 2,
//     with l the sum of the f16-rounded P that the PV MMA used (one row sum:
//     each normal f16 weight is within 2^-11 of its value, relative, so lse
//     moves by at most 4.9e-4 against the sum of unrounded terms, plus
//     2^-25 per subnormal weight below 2^-14).
// TMEM: FwdCfg (S, P, O of each tile).
#include "kernels.cuh"
#include "ptx.cuh"

namespace exattn {

template <int D>
struct FwdCfg {
  static constexpr int BM = 128;                   // query rows per tile (TMEM lanes)
  static constexpr int BN = 128;                   // keys per K/V tile
  static constexpr int NCHUNK = D / 64;            // 128-byte swizzle atoms across d
  static constexpr int CHUNK_BYTES = 128 * 128;    // 128 rows x 128 bytes
  static constexpr int TILE_BYTES = NCHUNK * CHUNK_BYTES;
  static constexpr int STAGES = (D == 64) ? 4 : 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + 2 * TILE_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_V + STAGES * TILE_BYTES;
  static constexpr int SMEM_BYTES = OFF_BAR + 512 + 1024;  // + barriers + alignment slack
  static_assert(SMEM_BYTES > 120 * 1024, "one CTA per SM: it holds all 512 TMEM columns");
  static constexpr int THREADS = 320;
  // TMEM.  d = 128: S_t at 128 t with P_t written over its first 64
  // columns, O_t at 256 + 128 t.  d = 64: S_t at 128 t, P_t in its own
  // columns 256 + 64 t, O_t at 384 + 64 t -- P apart from S lets the next
  // key tile's S_t be computed while the softmax still works on this one.
  static constexpr bool EARLY_S = D == 64;
  static constexpr uint32_t TM_COLS = 512;
  __host__ __device__ static constexpr uint32_t tm_s(int t) { return 128u * t; }
  __host__ __device__ static constexpr uint32_t tm_p(int t) { return EARLY_S ? 256u + 64u * t : 128u * t; }
  __host__ __device__ static constexpr uint32_t tm_o(int t) { return EARLY_S ? 384u + 64u * t : 256u + 128u * t; }
};

// Threads of the forward CTA: 8 softmax warps, the TMA warp and the MMA warp,
// plus two warps that convert V tiles to f16 when the inputs are bf16.
template <typename T>
struct FwdThreads {
  static constexpr bool kConvertV = Elem<T>::kFmt != Elem<__half>::kFmt;
  static constexpr int value = kConvertV ? 384 : 320;
};

template <int STAGES>
struct FwdBars {
  uint64_t q_full[2];
  uint64_t k_full[STAGES], k_empty[STAGES];
  uint64_t v_full[STAGES], v_empty[STAGES];
  uint64_t v_conv[STAGES];  // V tile converted to f16 (bf16 inputs only)
  uint64_t s_full[2];  // S_t ready (also: every earlier MMA of the CTA done)
  uint64_t s_free[2];  // d = 64: the softmax threads of tile t have loaded S_t
  uint64_t p_full[2];  // P_t written to TMEM by the 128 softmax threads
  uint64_t pv_done[2];  // d = 64: P_t V_j complete (P_t and O_t free)
  uint64_t o_full[2];  // last P_t V_j of tile t done
  uint64_t mma_done;   // every MMA of the CTA done (teardown)
  uint32_t tmem_base;
  int abort;
};

// Rescale threshold for the running max, in log2 units: P stays below 2^8.
constexpr float kRescaleThreshold = 8.0f;

// bf16 pair -> f16 pair, round to nearest even (exact in the f16 normal range).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  return pack_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

template <typename T, int D, bool CAUSAL, bool ONE_TILE>
__global__ void __launch_bounds__(FwdThreads<T>::value, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, T* __restrict__ out, Strides so,
                    float* __restrict__ lse_out, int N_max, int H, int BH, int n_pairs, int group, int window,
                    float scale_log2, SeqView seq, KvSplit kv, float* __restrict__ o32, unsigned* err) {
  using C = FwdCfg<D>;
  using E = Elem<T>;
  using PE = Elem<__half>;  // P and the converted V: the P V product runs in f16
  constexpr bool kConvertV = FwdThreads<T>::kConvertV;
  using Bars = FwdBars<C::STAGES>;
  static_assert(sizeof(Bars) <= 512, "barrier block too large");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::OFF_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  EXATTN_TRACE_INIT();

  // Heaviest work first: under the causal mask the last query pairs see the
  // most keys.  blockIdx = (group of heads, pair, key split, head in group).
  const GridPos gp = grid_pos(static_cast<int>(blockIdx.x), BH, n_pairs, kv.n_splits, group);
  const int pair = n_pairs - 1 - gp.tile;
  const int split = gp.sub;
  const int bh = gp.bh;
  const int hh = bh % H, bb = bh / H;  // head and batch index
  // A CTA owns two query tiles, or one (ONE_TILE: n_pairs then counts single
  // tiles and tile 1 stays empty) when two-tile CTAs would leave SMs idle.
  const int q0 = pair * (ONE_TILE ? 1 : 2) * C::BM;
  // This batch's rows (a packed variable-length batch may be shorter than the
  // grid's longest sequence: such a CTA has nothing to do).
  const SeqRows sr0 = seq_rows(seq, bb, hh, H, N_max);
  const int N = sr0.n, row0 = sr0.start, bt = sr0.b_coord;
  if (q0 >= N) return;
  // Keys: Nk of them, the queries aligned to the last N (query i at key
  // position i + off; off = 0 unless a decode-shaped call gave more keys).
  const int Nk = kv.nk > 0 ? kv.nk : N;
  const int off = Nk - N;
  // Keys any row of a query tile can see: up to its diagonal (causal) or
  // window - 1 past it (window W > 0: key j visible to query i iff
  // i + off - j < W, and also j - i - off < W without the causal mask), and
  // from the first row's window start.  Both tiles of the CTA stream key
  // tiles from the first tile of query tile 0 (kv_lo), tile 1 at most one
  // tile early, within this CTA's key split.
  auto key_end = [&](int t) {  // exclusive
    const int r0 = q0 + t * C::BM, r1 = min(N, r0 + C::BM);
    if (r0 >= N) return 0;
    if (CAUSAL) return min(Nk, r1 + off);
    return window > 0 ? min(Nk, r1 - 1 + off + window) : Nk;
  };
  const int split_lo = split * kv.tiles_per_split, split_hi = split_lo + kv.tiles_per_split;
  const int kv_lo = max(window > 0 ? max(0, q0 + off - window + 1) / C::BN : 0, split_lo);
  // Key tiles visited by query tile t, counted from kv_lo (0 if none).
  auto tiles_for = [&](int t) {
    const int e = key_end(t);
    return e == 0 ? 0 : max(0, min((e + C::BN - 1) / C::BN, split_hi) - kv_lo);
  };
  const int nkv0 = tiles_for(0), nkv1 = ONE_TILE ? 0 : tiles_for(1);
  const int n_iter = max(nkv0, nkv1);

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->q_full[t], 1);
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->s_free[t], 4);  // one arrival per softmax warp
      mbar_init(&bars->p_full[t], 4);
      mbar_init(&bars->pv_done[t], 1);
      mbar_init(&bars->o_full[t], 1);
    }
    mbar_init(&bars->mma_done, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->v_empty[s], 1);
      mbar_init(&bars->v_conv[s], 2);  // one arrival per converting warp
    }
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(&bars->tmem_base, C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const WaitCtl wc{&bars->abort, err};

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const uint64_t pol_kv = l2_policy_evict_last();   // K/V are re-read by every query pair of the head
      const uint64_t pol_q = l2_policy_evict_first();   // Q is read once
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if ((t == 0 ? nkv0 : nkv1) == 0) continue;
        mbar_arrive_expect_tx(&bars->q_full[t], C::TILE_BYTES);
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_4d(&tm_q, &bars->q_full[t], smem + C::OFF_Q + t * C::TILE_BYTES + c * C::CHUNK_BYTES, c * 64,
                      row0 + q0 + t * C::BM, hh, bt, pol_q);
      }
      int issued_k = 0, issued_v = 0;
      for (int j = 0; j < n_iter; ++j) {
        const int s = j % C::STAGES;
        const uint32_t ph = (j / C::STAGES) & 1;
        if (!mbar_wait(&bars->k_empty[s], ph ^ 1, wc)) break;
        EXATTN_TRACE_POINT(0, j, 0);
        mbar_arrive_expect_tx(&bars->k_full[s], C::TILE_BYTES);
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_4d(&tm_k, &bars->k_full[s], smem + C::OFF_K + s * C::TILE_BYTES + c * C::CHUNK_BYTES, c * 64,
                      row0 + (kv_lo + j) * C::BN, hh, bt, pol_kv);
        issued_k = j + 1;
        if (!mbar_wait(&bars->v_empty[s], ph ^ 1, wc)) break;
        EXATTN_TRACE_POINT(0, j, 1);
        mbar_arrive_expect_tx(&bars->v_full[s], C::TILE_BYTES);
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_4d(&tm_v, &bars->v_full[s], smem + C::OFF_V + s * C::TILE_BYTES + c * C::CHUNK_BYTES, c * 64,
                      row0 + (kv_lo + j) * C::BN, hh, bt, pol_kv);
        issued_v = j + 1;
      }
      if (*reinterpret_cast<volatile int*>(&bars->abort)) {
        // Never leave a copy in flight into shared memory this CTA is about to release.
        for (int t = 0; t < 2; ++t)
          if ((t == 0 ? nkv0 : nkv1) > 0) mbar_wait_drain(&bars->q_full[t], 0, err);
        for (int j = max(0, issued_k - C::STAGES); j < issued_k; ++j)
          mbar_wait_drain(&bars->k_full[j % C::STAGES], (j / C::STAGES) & 1, err);
        for (int j = max(0, issued_v - C::STAGES); j < issued_v; ++j)
          mbar_wait_drain(&bars->v_full[j % C::STAGES], (j / C::STAGES) & 1, err);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop (waits and descriptor arithmetic stay
    // warp-uniform); the elected lane issues the tcgen05 instructions.
    constexpr uint32_t idesc_s = idesc_f16kind(E::kFmt, 128, C::BN, 0, 0);  // Q, K both K-major
    constexpr uint32_t idesc_o = idesc_f16kind(PE::kFmt, 128, D, 0, 1);     // f16 P from TMEM, f16 V MN-major
    const uint64_t q_desc = sdesc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
    const uint64_t k_desc = sdesc_sw128(smem_u32(smem + C::OFF_K), 16, 1024);
    const uint64_t v_desc = sdesc_sw128(smem_u32(smem + C::OFF_V), C::CHUNK_BYTES, 1024);
    constexpr uint32_t kTileDesc = C::TILE_BYTES >> 4;  // descriptor units are 16 bytes

    auto issue_s = [&](int t, int stage) {
      const uint64_t a = q_desc + t * kTileDesc, b = k_desc + stage * kTileDesc;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32) >> 4;
        mma_ss(tmem + C::tm_s(t), a + off, b + off, idesc_s, kk > 0);
      }
    };
    auto issue_pv = [&](int t, int stage, bool acc) {
      const uint64_t b = v_desc + stage * kTileDesc;
#pragma unroll
      for (int kk = 0; kk < C::BN / 16; ++kk)
        mma_ts(tmem + C::tm_o(t), tmem + C::tm_p(t) + kk * 8, b + ((kk * 16 * 128) >> 4), idesc_o,
               (acc || kk > 0) ? 1u : 0u);
    };
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, wc));
    };

    bool ok = true;
    if (nkv0 > 0) ok = wait_all(&bars->q_full[0], 0);
    if (ok && nkv1 > 0) ok = wait_all(&bars->q_full[1], 0);
    if (ok && n_iter > 0) ok = wait_all(&bars->k_full[0], 0);
    if (ok && n_iter > 0) {
      tc_fence_after();
      if (elect_one()) {
        if (nkv0 > 0) {
          issue_s(0, 0);
          mma_commit(&bars->s_full[0]);
        }
        if (nkv1 > 0) {
          issue_s(1, 0);
          mma_commit(&bars->s_full[1]);
        }
        mma_commit(&bars->k_empty[0]);
      }
      __syncwarp();
    }
    if constexpr (C::EARLY_S) {
      // Per key step j: the next scores S_t(j+1) as soon as tile t's softmax
      // has loaded S_t(j) (its P goes to separate columns), then P_t V_j.
      for (int j = 0; ok && j < n_iter; ++j) {
        const int s = j % C::STAGES;
        const uint32_t ph = (j / C::STAGES) & 1;
        const int s1 = (j + 1) % C::STAGES;
        const uint32_t ph1 = ((j + 1) / C::STAGES) & 1;
        bool k_ready = false, v_ready = false;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int nkv_t = t == 0 ? nkv0 : nkv1;
          if (!ok || j + 1 >= nkv_t) continue;
          if (!(ok = wait_all(&bars->s_free[t], j & 1))) continue;
          if (!k_ready) {
            if (!(ok = wait_all(&bars->k_full[s1], ph1))) continue;
            k_ready = true;
          }
          tc_fence_after();
          if (elect_one()) {
            issue_s(t, s1);
            mma_commit(&bars->s_full[t]);
          }
          __syncwarp();
        }
        if (k_ready) {
          if (elect_one()) mma_commit(&bars->k_empty[s1]);
          __syncwarp();
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int nkv_t = t == 0 ? nkv0 : nkv1;
          if (!ok || j >= nkv_t) continue;
          if (!(ok = wait_all(&bars->p_full[t], j & 1))) continue;
          if (!v_ready) {
            if (!(ok = wait_all(kConvertV ? &bars->v_conv[s] : &bars->v_full[s], ph))) continue;
            v_ready = true;
          }
          tc_fence_after();
          if (elect_one()) {
            issue_pv(t, s, j > 0);
            mma_commit(&bars->pv_done[t]);
            if (t == 1 || nkv1 <= j) mma_commit(&bars->v_empty[s]);
            if (j + 1 == nkv_t) mma_commit(&bars->o_full[t]);
          }
          __syncwarp();
        }
      }
    } else {
      for (int j = 0; ok && j < n_iter; ++j) {
        const int s = j % C::STAGES;
        const uint32_t ph = (j / C::STAGES) & 1;
        const int s1 = (j + 1) % C::STAGES;
        const uint32_t ph1 = ((j + 1) / C::STAGES) & 1;
        bool v_ready = false, k_ready = false;
  #pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int nkv_t = t == 0 ? nkv0 : nkv1;
          if (!ok || j >= nkv_t) continue;
          if (!(ok = wait_all(&bars->p_full[t], j & 1))) continue;
          if (lane == 0) EXATTN_TRACE_POINT(1, j, 4 * t + 0);
          if (!v_ready) {
            if (!(ok = wait_all(kConvertV ? &bars->v_conv[s] : &bars->v_full[s], ph))) continue;
            v_ready = true;
          }
          if (lane == 0) EXATTN_TRACE_POINT(1, j, 4 * t + 1);
          tc_fence_after();
          if (elect_one()) {
            issue_pv(t, s, j > 0);
            // V_j is free once the last tile's P V_j is done; releasing it here,
            // inside the block, keeps the block boundary free of commits.
            if (t == 1 || nkv1 <= j) mma_commit(&bars->v_empty[s]);
          }
          __syncwarp();
          if (j + 1 < nkv_t) {
            if (!k_ready) {
              if (!(ok = wait_all(&bars->k_full[s1], ph1))) continue;
              k_ready = true;
              tc_fence_after();
            }
            if (lane == 0) EXATTN_TRACE_POINT(1, j, 4 * t + 2);
            if (elect_one()) {
              issue_s(t, s1);
              mma_commit(&bars->s_full[t]);
            }
            __syncwarp();
            if (lane == 0) EXATTN_TRACE_POINT(1, j, 4 * t + 3);
          } else {
            if (elect_one()) mma_commit(&bars->o_full[t]);
            __syncwarp();
          }
        }
        if (k_ready) {
          if (elect_one()) mma_commit(&bars->k_empty[s1]);
          __syncwarp();
        }
      }
    }
    // Nothing may still read shared memory or write TMEM once the CTA tears down.
    if (elect_one()) mma_commit(&bars->mma_done);
    __syncwarp();
    if (lane == 0) mbar_wait_drain(&bars->mma_done, 0, err);
    __syncwarp();
  } else if (warp >= 10) {
    // ------------------------------------------------------------ V to f16 (bf16 inputs)
    // 64 threads convert each landed V tile in place (the layout is the same
    // for both 16-bit types), then make their generic-proxy stores visible to
    // the tensor core's async-proxy reads before arriving.
    if constexpr (kConvertV) {
      constexpr int NVEC = C::TILE_BYTES / 16;  // 16-byte vectors per tile
      constexpr int PER = NVEC / 64, BATCH = 8;
      static_assert(PER % BATCH == 0, "conversion batches must divide the tile");
      const int ct = (warp - 10) * 32 + lane;
      for (int j = 0; j < n_iter; ++j) {
        const int s = j % C::STAGES;
        if (!mbar_wait_warp(&bars->v_full[s], (j / C::STAGES) & 1, wc)) break;
        uint4* tile = reinterpret_cast<uint4*>(smem + C::OFF_V + s * C::TILE_BYTES);
#pragma unroll 1
        for (int b0 = 0; b0 < PER; b0 += BATCH) {
          uint4 x[BATCH];
#pragma unroll
          for (int u = 0; u < BATCH; ++u) x[u] = tile[(b0 + u) * 64 + ct];
#pragma unroll
          for (int u = 0; u < BATCH; ++u)
            tile[(b0 + u) * 64 + ct] = make_uint4(bf16x2_to_f16x2(x[u].x), bf16x2_to_f16x2(x[u].y),
                                                  bf16x2_to_f16x2(x[u].z), bf16x2_to_f16x2(x[u].w));
        }
        fence_proxy_async_smem();
        mbar_arrive_warp(&bars->v_conv[s]);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;          // query row within the tile == TMEM lane
    const int row_g = q0 + t * C::BM + row;  // query row within the head
    const uint32_t lane_bits = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_bits + C::tm_s(t);
    const uint32_t tP = tmem + lane_bits + C::tm_p(t);
    const uint32_t tO = tmem + lane_bits + C::tm_o(t);
    float m_ref = -INFINITY;  // reference max, log2 units of the scaled logits
    float lb = 0.f;           // running sum of the f16-rounded 2^(x - m_ref) the PV MMA uses
    bool ok = true;  // cleared only by a wait that gave up
    for (int j = 0; ok && j < (t == 0 ? nkv0 : nkv1); ++j) {
      if (!(ok = mbar_wait_warp(&bars->s_full[t], j & 1, wc))) break;
      if (row == 0) EXATTN_TRACE_POINT(2 + t, j, 0);
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + c * 32, sr[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_reg_fence(sr[c]);
      if constexpr (C::EARLY_S) {
        // S_t is in registers: the MMA warp may compute the next one over it.
        tc_fence_before();
        mbar_arrive_warp(&bars->s_free[t]);
      }

      const int kv0 = (kv_lo + j) * C::BN;
      const int tr0 = q0 + t * C::BM;  // first row of this query tile
      // Some key of this tile is hidden from some row of the query tile: past
      // the diagonal, past N, or outside a row's window.
      const bool need_mask = (CAUSAL && kv0 + C::BN - 1 > tr0 + off) || (kv0 + C::BN > Nk) ||
                             (window > 0 && (kv0 < tr0 + off + C::BM - window ||
                                             (!CAUSAL && kv0 + C::BN - 1 > tr0 + off + window - 1)));
      if (need_mask) {
        const int pos = row_g + off;  // this row's key position
        int lim = Nk - kv0;           // visible columns c: lo <= c < lim
        if (CAUSAL) lim = min(lim, pos - kv0 + 1);
        else if (window > 0) lim = min(lim, pos + window - kv0);
        const int lo = window > 0 ? pos - window + 1 - kv0 : 0;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (c * 32 + e >= lim || c * 32 + e < lo) sr[c][e] = __float_as_uint(-INFINITY);
      }
      // Row max as eight independent chains of three-input maxima: the
      // reduction is exact in any order, and a short chain keeps the
      // warpgroup's latency (which the tensor core waits on) low.
      float mx;
      {
        auto x = [&](int f) { return __uint_as_float(sr[f >> 5][f & 31]); };
        float pm[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) pm[k] = fmaxf(x(k), x(k + 8));
#pragma unroll
        for (int f = 16; f < 128; f += 16)
#pragma unroll
          for (int k = 0; k < 8; ++k) pm[k] = fmax3(pm[k], x(f + k), x(f + 8 + k));
        mx = fmax3(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7]));
      }
      const float m_new = fmaxf(m_ref, mx * scale_log2);
      // Move the reference max only when it grew by more than the threshold.
      float alpha = 1.f;
      bool rescale_warp = false;
      if (j == 0) {
        m_ref = m_new;
      } else {
        const bool need = m_new > m_ref + kRescaleThreshold;
        rescale_warp = __any_sync(0xffffffffu, need);
        if (need) {
          alpha = ex2(m_ref - m_new);
          m_ref = m_new;
        }
      }
      // A row that has seen only masked keys so far (a window start inside a
      // later tile) keeps m_ref = -inf: its P is 0, never NaN.
      const float neg_m = m_ref == -INFINITY ? 0.f : -m_ref;
      const float2 sc2 = make_float2(scale_log2, scale_log2), nm2 = make_float2(neg_m, neg_m);
      uint32_t pk[4][16];  // P as f16 pairs, kept for the rounded sum below
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float2 y = ffma2(make_float2(__uint_as_float(sr[c][2 * e]), __uint_as_float(sr[c][2 * e + 1])), sc2, nm2);
          const float2 p = make_float2(ex2(y.x), ex2(y.y));
          pk[c][e] = PE::pack(p.x, p.y);
        }
        if constexpr (!C::EARLY_S) tmem_st16(tP + c * 16, pk[c]);  // P_t over the first 64 columns of S_t
      }
      if constexpr (C::EARLY_S) {
        // Only now must P_t(j-1) V_{j-1} be done (its P_t columns and the O_t
        // row are written next): the maxima and exponentials above ran while
        // the tensor core worked on it.
        if (j > 0 && !(ok = mbar_wait_warp(&bars->pv_done[t], (j - 1) & 1, wc))) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_st16(tP + c * 16, pk[c]);  // P_t in its own columns
      }
      if (rescale_warp) {
        // P_t(j-1) V_{j-1} has completed (d = 128: S_t(j) is issued after it;
        // d = 64: pv_done waited above): the O row is stable.  This branch is
        // rare; at d = 128 it runs rolled, which keeps the kernel inside its
        // 168 registers without spills.
#pragma unroll(D == 128 ? 1 : D / 32)
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o_r[32];
          tmem_ld32(tO + c * 32, o_r);
          tmem_wait_ld();
          tmem_reg_fence(o_r);
#pragma unroll
          for (int e = 0; e < 32; ++e) o_r[e] = __float_as_uint(__uint_as_float(o_r[e]) * alpha);
          tmem_st32(tO + c * 32, o_r);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      if (row == 0) EXATTN_TRACE_POINT(2 + t, j, 1);
      mbar_arrive_warp(&bars->p_full[t]);
      // O is normalised by the sum of the f16-rounded weights the PV MMA
      // used: a row dominated by a few keys then keeps an exact convex
      // combination of V rows instead of inheriting their rounding.  Done
      // after the hand-off, off the tensor core's critical path.
      float2 rb[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 16; ++e) rb[e & 1] = PE::add_pair(pk[c][e], rb[e & 1]);
      const float2 rbs = fadd2(rb[0], rb[1]);
      lb = lb * alpha + (rbs.x + rbs.y);
    }
    // ---------------------------------------------------------- epilogue
    const bool any = (t == 0 ? nkv0 : nkv1) > 0;
    if (ok && any) ok = mbar_wait_warp(&bars->o_full[t], 0, wc);
    if (ok && kv.part_o) {
      // Key split: this split's O (normalised within it) and both
      // logsumexps in fp32; a row that saw no key here gets O = 0 and -inf.
      const long long prow = (static_cast<long long>(split) * BH + bh) * kv.nq_pad + row_g;
      float* po = kv.part_o + prow * D;
      const float inv_l = lb > 0.f ? 1.f / lb : 0.f;
      if (any) tc_fence_after();
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o_r[32];
        if (any) {
          tmem_ld32(tO + c * 32, o_r);
          tmem_wait_ld();
          tmem_reg_fence(o_r);
        }
        if (row_g < N) {
          float4* dst = reinterpret_cast<float4*>(po + c * 32);
#pragma unroll
          for (int v4 = 0; v4 < 8; ++v4)
            dst[v4] = any ? make_float4(__uint_as_float(o_r[4 * v4]) * inv_l, __uint_as_float(o_r[4 * v4 + 1]) * inv_l,
                                        __uint_as_float(o_r[4 * v4 + 2]) * inv_l,
                                        __uint_as_float(o_r[4 * v4 + 3]) * inv_l)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      if (row_g < N) {
        kv.part_lse[prow] = lb > 0.f ? (m_ref + log2f(lb)) * 0.6931471805599453f : -INFINITY;
        kv.part_lseb[prow] = lb > 0.f ? (m_ref + log2f(lb)) * 0.6931471805599453f : -INFINITY;
      }
    } else if (ok && any) {
      tc_fence_after();
      const float inv_l = 1.f / lb;
      T* orow = out + bt * so.b + hh * so.h + static_cast<long long>(row0 + row_g) * so.n;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o_r[32];
        tmem_ld32(tO + c * 32, o_r);
        tmem_wait_ld();
        tmem_reg_fence(o_r);
        if (row_g < N) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = E::pack(__uint_as_float(o_r[2 * e]) * inv_l, __uint_as_float(o_r[2 * e + 1]) * inv_l);
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
          if (o32 != nullptr) {
            // The same row before rounding to the output type, for a backward
            // that takes D_i = dO_i . O_i from it.
            float4* dst32 = reinterpret_cast<float4*>(o32 + (static_cast<long long>(bh) * N_max + row_g) * D + c * 32);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              dst32[v4] = make_float4(__uint_as_float(o_r[4 * v4]) * inv_l, __uint_as_float(o_r[4 * v4 + 1]) * inv_l,
                                      __uint_as_float(o_r[4 * v4 + 2]) * inv_l,
                                      __uint_as_float(o_r[4 * v4 + 3]) * inv_l);
          }
        }
      }
      if (row_g < N) lse_out[sr0.stat0 + row_g] = (m_ref + log2f(lb)) * 0.6931471805599453f;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, C::TM_COLS);
}

template <typename T, int D, bool CAUSAL>
static cudaError_t launch_fwd_t(const FwdArgs& a, cudaStream_t stream) {
  using C = FwdCfg<D>;
  cudaError_t e;
  KvSplit kv = a.kv;
  if (kv.n_splits < 1) {  // one CTA covers all keys of its query pair
    kv.n_splits = 1;
    kv.tiles_per_split = 1 << 30;
  }
  // Two query tiles per CTA share each K/V tile and hide each other's
  // hand-offs.  When even one tile per CTA fits in one wave of SMs (small
  // problems), one tile per CTA halves the longest CTA's chain (B1 H2 N256:
  // 0.0133 -> 0.0109 ms); at 128 pairs it gained nothing, and in the host
  // pipeline, whose head groups share the SMs on two streams, it cost 6 %.
  int sms = 0;
  e = note_cuda(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, a.device), "cudaDeviceGetAttribute");
  if (e != cudaSuccess) return e;
  const int pairs = (a.N + 2 * C::BM - 1) / (2 * C::BM);
  const bool one_tile = kv.n_splits == 1 && 2ll * pairs * a.BH <= sms;
  const int n_pairs = one_tile ? (a.N + C::BM - 1) / C::BM : pairs;
  auto kern = one_tile ? attn_fwd_kernel<T, D, CAUSAL, true> : attn_fwd_kernel<T, D, CAUSAL, false>;
  e = ensure_smem_attr(reinterpret_cast<const void*>(kern), C::SMEM_BYTES, a.device);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(n_pairs) * kv.n_splits * a.BH;
  // Group heads so their K and V stay in L2 -- except when the key splits read
  // disjoint key ranges (nothing is re-read across CTAs) or the packed
  // sequences differ in length (plain heaviest-first order balances them
  // better; measured).  A group's K, V fill a quarter of L2: with half, the
  // B4 H32 N4096 d64 forward fetched K and V about three times (523-560 MB
  // per launch), with a quarter once (257 MB; 270.5 MB algorithmic), in the
  // same time.
  const int group = (kv.n_splits > 1 || a.seq.cu_seqlens)
                        ? a.BH
                        : l2_group(2ll * (kv.nk > 0 ? kv.nk : a.N) * D * static_cast<long long>(sizeof(T)), a.BH,
                                   kL2GroupBytes / 2);
  kern<<<static_cast<unsigned>(grid), FwdThreads<T>::value, C::SMEM_BYTES, stream>>>(
      *a.tm_q, *a.tm_k, *a.tm_v, static_cast<T*>(a.o), a.so, a.lse, a.N, a.H, a.BH, n_pairs, group, a.window,
      a.scale_log2, a.seq, kv, a.o32, a.err);
  return note_cuda(cudaGetLastError(), "forward kernel launch");
}

template <typename T>
static cudaError_t launch_fwd_dt(const FwdArgs& a, cudaStream_t stream) {
  if (a.d == 64) return a.causal ? launch_fwd_t<T, 64, true>(a, stream) : launch_fwd_t<T, 64, false>(a, stream);
  return a.causal ? launch_fwd_t<T, 128, true>(a, stream) : launch_fwd_t<T, 128, false>(a, stream);
}

cudaError_t launch_fwd(const FwdArgs& a, cudaStream_t stream) {
  return a.dtype == kF16 ? launch_fwd_dt<__half>(a, stream) : launch_fwd_dt<__nv_bfloat16>(a, stream);
}

}  // namespace exattn
