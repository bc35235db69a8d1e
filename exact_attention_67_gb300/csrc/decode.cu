// decode.cu -- the decode-shaped forward for a few queries against many keys
// (at d = 128, Nq <= 12 query rows per (batch, head), queries at the last Nq
// key positions), for sm_103a.
//
// The forward kernel runs a 128-row query tile per MMA; with one to sixteen
// real query rows that wastes the products and a 128-row softmax on every
// key step.  Here the keys take the MMA's M side instead (the tiling and the
// online softmax of "Gemini 3 Flash的注意力内核重写：算子融合如何实现亚毫秒级推理",
// §2 分块（Tiling）优化 and §3 在线softmax算法, with the roles of the two
// operands exchanged):
//   * S^T = K_j Q^T: M = 128 keys (TMEM lanes), N = 16 query columns, K = d;
//   * the online softmax runs down each query column: every thread holds one
//     key's 16 scores; a column's reference max moves only when a score
//     beats it by 2^8 (or the column sees its first key), so a step first
//     trades one bit per column between the four warps, and only a step
//     that needs it reduces the column maxima across the warpgroup;
//   * O^T += V_j^T P^T: M = d = 128 rows (TMEM lanes), N = 16, K = 128 keys,
//     with P^T written by the elementwise threads into shared memory in f16;
//   * the epilogue reads O^T row d of every query column from lane d, so the
//     output rows are written with consecutive threads on consecutive d.
// Keys are split over CTAs (as in the forward's key split) and the splits'
// fp32 partial O and logsumexps are combined by the split-merge kernel (merge.cu).
// Measured against the forward kernel's key-split path on the same GPU (B8
// H16 Nk16384 and B4 H32 Nk32768, d = 128): 1.26x faster for Nq <= 4,
// 1.17x at 8, 1.07-1.10x at 12, slower at 16 (the per-key column work
// grows with Nq while the forward's softmax runs along rows); at d = 64 a
// step moves half the bytes for the same column work and the kernel was
// slower for every Nq.  Hence the d = 128, Nq <= 12 dispatch in the C ABI.
//
// CTA: warps 0-3 elementwise (thread = key row of S^T and row d of O^T),
// warp 4 TMA producer, warp 5 MMA issuer, and for bf16 inputs warps 6-7
// convert each V tile to f16 in place.  The four elementwise warps trade
// their column maxima through shared memory behind a named barrier that
// every one of them passes once per key step, also after a bounded wait has
// given up (the work is skipped then, the barrier never).  TMEM: two S^T
// buffers of 16 columns and O^T (16 columns), 64 columns allocated.
// Precision as in the forward: P rounded to f16 for the P V product (V tiles
// converted to f16 in shared memory for bf16 inputs), the row sums formed
// from the f16-rounded weights, fp32 accumulation.
#include "kernels.cuh"
#include "ptx.cuh"

namespace exattn {

namespace {

template <int D>
struct DecCfg {
  static_assert(D == 128, "the decode kernel is dispatched at d = 128 only");
  static constexpr int BN = 128;                // keys per step (TMEM lanes of S^T)
  static constexpr int NQ = kDecodeQCols;       // query columns (the MMA's N; queries past Nq are zero rows of Q)
  static constexpr int NCHUNK = D / 64;         // 128-byte swizzle atoms across d
  static constexpr int KV_CHUNK = BN * 128;     // one 64-column chunk of a 128-row tile
  static constexpr int KV_TILE = NCHUNK * KV_CHUNK;
  static constexpr int Q_CHUNK = NQ * 128;      // one 64-column chunk of the 16-row Q tile
  static constexpr int Q_TILE = NCHUNK * Q_CHUNK;
  static constexpr int P_CHUNK = NQ * 128;      // P^T: 16 rows x 64 keys (f16)
  static constexpr int P_TILE = 2 * P_CHUNK;    // 128 keys
  // One CTA per SM with three stages of K and V (192 KB) in flight.
  static constexpr int STAGES = 3;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + STAGES * KV_TILE;
  static constexpr int OFF_Q = OFF_V + STAGES * KV_TILE;
  static constexpr int OFF_P = OFF_Q + Q_TILE;             // two P^T buffers
  // Column maxima [2][4 warps][16] and sums [4][16] (floats), then the
  // warps' need-a-new-max bits [2][4] (32-bit words).
  static constexpr int OFF_RED = OFF_P + 2 * P_TILE;
  static constexpr int OFF_BAR = OFF_RED + 3 * 4 * NQ * 4 + 2 * 4 * 4;
  static constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;  // + barriers + alignment slack
  static_assert(SMEM_BYTES <= 232448, "over the 227 KB shared-memory limit");
  static constexpr int PRODUCER_WARP = 4, MMA_WARP = 5;
  static constexpr uint32_t TM_S = 0, TM_O = 2 * NQ, TM_COLS = 64;  // S^T buffer b at 16 b
};

// Threads: four elementwise warps, the producer and the MMA warp, plus two
// warps that convert V tiles to f16 when the inputs are bf16.
template <typename T>
struct DecThreads {
  static constexpr bool kConvertV = Elem<T>::kFmt != Elem<__half>::kFmt;
  static constexpr int value = kConvertV ? 256 : 192;
};

template <int STAGES>
struct DecBars {
  uint64_t q_full;
  uint64_t kv_full[STAGES], kv_empty[STAGES];
  uint64_t s_full[2], s_free[2];  // S^T buffer b: written by the MMA / read by the elementwise threads
  uint64_t p_full[2], p_free[2];  // P^T buffer b: written by the elementwise threads / read by P V
  uint64_t v_conv[STAGES];        // V tile converted to f16 (bf16 inputs only)
  uint64_t pv_done;               // each step's P V complete
  uint64_t o_full;                // the last P V complete
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

// Reference max moves only when a column's max grew by more than this
// (log2 units): the weights stay below 2^8.
constexpr float kDecRescale = 8.0f;

// bf16 pair -> f16 pair, round to nearest even (exact in the f16 normal range).
__device__ __forceinline__ uint32_t dec_bf16x2_to_f16x2(uint32_t w) {
  return pack_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// As tmem_reg_fence, for a 16-register TMEM load.
__device__ __forceinline__ void reg_fence16(uint32_t (&r)[16]) {
  asm volatile("" : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
               "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
               "+r"(r[14]), "+r"(r[15]));
}

}  // namespace

template <typename T, int D, bool CAUSAL>
__global__ void __launch_bounds__(DecThreads<T>::value, 1)
    attn_decode_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, T* __restrict__ out, Strides so,
                       float* __restrict__ lse_out, int Nq, int Nk, int H, int BH, int window, float scale_log2,
                       KvSplit kv, unsigned* err) {
  using C = DecCfg<D>;
  using E = Elem<T>;
  using PE = Elem<__half>;  // P and the converted V: the P V product runs in f16
  using Bars = DecBars<C::STAGES>;
  constexpr bool kConvertV = DecThreads<T>::kConvertV;
  constexpr int NQ = C::NQ, BN = C::BN;
  static_assert(sizeof(Bars) <= 256, "barrier block too large");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::OFF_BAR);
  float* red = reinterpret_cast<float*>(smem + C::OFF_RED);  // [2][4][NQ] maxima, then [4][NQ] sums
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Grid: (batch, head) major, key split minor.  The split covers key tiles
  // [split tps, (split + 1) tps), cut to the tiles some query can see: with a
  // window, none before the first query's window start (query q sits at key
  // position Nk - Nq + q).
  const int n_splits = kv.n_splits;
  const int bh = static_cast<int>(blockIdx.x) / n_splits, split = static_cast<int>(blockIdx.x) % n_splits;
  const int hh = bh % H, bb = bh / H;
  const int off = Nk - Nq;
  const int nkt = (Nk + BN - 1) / BN;
  const int vis_lo = window > 0 ? max(0, off - window + 1) / BN : 0;
  const int t_lo = max(split * kv.tiles_per_split, vis_lo);
  const int t_hi = min(nkt, (split + 1) * kv.tiles_per_split);
  const int ntiles = max(0, t_hi - t_lo);

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
      mbar_init(&bars->v_conv[s], 2);  // one arrival per converting warp
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->s_free[b], 4);   // one arrival per elementwise warp
      mbar_init(&bars->p_full[b], 4);
      mbar_init(&bars->p_free[b], 1);
    }
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == C::MMA_WARP) {
    tmem_alloc(&bars->tmem_base, C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The split merge, launched as this grid's programmatic dependent, may be
  // scheduled once every CTA has started; it waits for this grid's completion
  // before it reads anything.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const uint32_t tmem = bars->tmem_base;
  const WaitCtl wc{&bars->abort, err};

  if (warp == C::PRODUCER_WARP) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const uint64_t pol = l2_policy_evict_first();  // every byte is read by this CTA alone
      if (ntiles > 0) {
        // Q rows Nq..15 lie past the map's extent: TMA fills them with zeros.
        mbar_arrive_expect_tx(&bars->q_full, C::Q_TILE);
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_4d(&tm_q, &bars->q_full, smem + C::OFF_Q + c * C::Q_CHUNK, c * 64, 0, hh, bb, pol);
      }
      int issued = 0;
      for (int j = 0; j < ntiles; ++j) {
        const int s = j % C::STAGES;
        const uint32_t ph = (j / C::STAGES) & 1;
        if (!mbar_wait(&bars->kv_empty[s], ph ^ 1, wc)) break;
        mbar_arrive_expect_tx(&bars->kv_full[s], 2 * C::KV_TILE);
        const int row = (t_lo + j) * BN;
        for (int c = 0; c < C::NCHUNK; ++c) {
          tma_load_4d(&tm_k, &bars->kv_full[s], smem + C::OFF_K + s * C::KV_TILE + c * C::KV_CHUNK, c * 64, row, hh,
                      bb, pol);
          tma_load_4d(&tm_v, &bars->kv_full[s], smem + C::OFF_V + s * C::KV_TILE + c * C::KV_CHUNK, c * 64, row, hh,
                      bb, pol);
        }
        issued = j + 1;
      }
      if (*reinterpret_cast<volatile int*>(&bars->abort)) {
        // Never leave a copy in flight into shared memory this CTA is about to release.
        if (ntiles > 0) mbar_wait_drain(&bars->q_full, 0, err);
        for (int j = max(0, issued - C::STAGES); j < issued; ++j)
          mbar_wait_drain(&bars->kv_full[j % C::STAGES], (j / C::STAGES) & 1, err);
      }
    }
    __syncwarp();
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    // Per step j: S^T_j = K_j Q^T into TMEM buffer j % 2, then P^T V of step
    // j - 1 (its weights came back from the elementwise threads meanwhile).
    constexpr uint32_t idesc_s = idesc_f16kind(E::kFmt, 128, NQ, 0, 0);   // K, Q both K-major
    constexpr uint32_t idesc_o = idesc_f16kind(PE::kFmt, 128, NQ, 1, 0);  // V^T MN-major, P^T K-major
    const uint64_t q_desc = sdesc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
    const uint64_t k_desc = sdesc_sw128(smem_u32(smem + C::OFF_K), 16, 1024);
    const uint64_t p_desc = sdesc_sw128(smem_u32(smem + C::OFF_P), 16, 1024);
    // V^T of stage s as the MN-major A operand: its two 64-row groups along d
    // are the tile's 64-column chunks.
    auto v_desc = [&](int s) {
      return sdesc_sw128(smem_u32(smem + C::OFF_V + s * C::KV_TILE), C::KV_CHUNK, 1024);
    };
    auto wait_all = [&](uint64_t* bar, uint32_t parity) { return mbar_wait_warp(bar, parity, wc); };
    bool ok = ntiles == 0 || wait_all(&bars->q_full, 0);
    for (int j = 0; ok && j <= ntiles && ntiles > 0; ++j) {
      if (j < ntiles) {
        const int s = j % C::STAGES, b = j & 1;
        if (!(ok = wait_all(&bars->kv_full[s], (j / C::STAGES) & 1))) break;
        // Buffer b held S^T of step j - 2: the elementwise threads have loaded it.
        if (j >= 2 && !(ok = wait_all(&bars->s_free[b], ((j - 2) >> 1) & 1))) break;
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ko = ((kk >> 2) * C::KV_CHUNK + (kk & 3) * 32) >> 4;
            const uint32_t qo = ((kk >> 2) * C::Q_CHUNK + (kk & 3) * 32) >> 4;
            mma_ss(tmem + C::TM_S + b * NQ, k_desc + ((s * C::KV_TILE) >> 4) + ko, q_desc + qo, idesc_s, kk > 0);
          }
          mma_commit(&bars->s_full[b]);
        }
        __syncwarp();
      }
      if (j >= 1) {
        const int jp = j - 1, sp = jp % C::STAGES, bp = jp & 1;
        if (!(ok = wait_all(&bars->p_full[bp], (jp >> 1) & 1))) break;
        if (kConvertV && !(ok = wait_all(&bars->v_conv[sp], (jp / C::STAGES) & 1))) break;
        tc_fence_after();
        if (elect_one()) {
          const uint64_t vd = v_desc(sp);
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk) {
            const uint32_t po = ((kk >> 2) * C::P_CHUNK + (kk & 3) * 32) >> 4;
            mma_ss(tmem + C::TM_O, vd + ((kk * 16 * 128) >> 4), p_desc + ((bp * C::P_TILE) >> 4) + po, idesc_o,
                   (jp > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(&bars->pv_done);
          mma_commit(&bars->kv_empty[sp]);  // K_jp, V_jp read
          mma_commit(&bars->p_free[bp]);
          if (jp == ntiles - 1) mma_commit(&bars->o_full);
        }
        __syncwarp();
      }
    }
    // Nothing may still read shared memory or write TMEM once the CTA tears down.
    if (elect_one()) mma_commit(&bars->mma_done);
    __syncwarp();
    if (lane == 0) mbar_wait_drain(&bars->mma_done, 0, err);
    __syncwarp();
  } else if (warp >= 6) {
    // ------------------------------------------------------------ V to f16 (bf16 inputs)
    // 64 threads convert each landed V tile in place, then make their
    // generic-proxy stores visible to the tensor core's reads before arriving.
    if constexpr (kConvertV) {
      const int ct = (warp - 6) * 32 + lane;
      for (int j = 0; j < ntiles; ++j) {
        const int s = j % C::STAGES;
        if (!mbar_wait_warp(&bars->kv_full[s], (j / C::STAGES) & 1, wc)) break;
        uint4* tile = reinterpret_cast<uint4*>(smem + C::OFF_V + s * C::KV_TILE);
#pragma unroll 8
        for (int i = 0; i < C::KV_TILE / 16 / 64; ++i) {
          const uint4 x = tile[i * 64 + ct];
          tile[i * 64 + ct] = make_uint4(dec_bf16x2_to_f16x2(x.x), dec_bf16x2_to_f16x2(x.y),
                                         dec_bf16x2_to_f16x2(x.z), dec_bf16x2_to_f16x2(x.w));
        }
        fence_proxy_async_smem();
        mbar_arrive_warp(&bars->v_conv[s]);
      }
    }
  } else {
    // ------------------------------------------------------------ elementwise (thread = key row / d row)
    const int tid = threadIdx.x;  // 0..127: TMEM lane
    const uint32_t lane_bits = static_cast<uint32_t>(warp * 32) << 16;
    float m_ref[NQ], lsum[NQ];  // per query column: reference max (log2 units), this thread's weight sum
#pragma unroll
    for (int q = 0; q < NQ; ++q) {
      m_ref[q] = -INFINITY;
      lsum[q] = 0.f;
    }
    bool ok = true;
    // Every warp runs all ntiles steps and passes the step's named barrier
    // (id 1, the 128 elementwise threads) once, whatever its waits returned:
    // after a wait gives up, the work is skipped and the barrier still met.
    for (int j = 0; j < ntiles; ++j) {
      const int b = j & 1;
      float x[NQ];
      float* rb = red + b * 4 * NQ;  // the four warps' column maxima, buffer j % 2
      uint32_t need = 0;             // bit q: column q's reference max must move
      if (ok) ok = mbar_wait_warp(&bars->s_full[b], (j >> 1) & 1, wc);
      if (ok) {
        tc_fence_after();
        uint32_t sv[NQ];
        tmem_ld16(tmem + lane_bits + C::TM_S + b * NQ, sv);
        tmem_wait_ld();
        reg_fence16(sv);
        tc_fence_before();
        mbar_arrive_warp(&bars->s_free[b]);  // the MMA warp may compute S^T_{j+2} into buffer b
        // Scaled logits of this thread's key for each query column; hidden
        // ones (and columns past Nq, within the last group of four) -inf.
        // Per-element masks only on tiles where some query cannot see some
        // key: past Nk, past the diagonal, or outside a window.
        const int kj0 = (t_lo + j) * BN, kj = kj0 + tid;
        const bool need_mask = kj0 + BN > Nk || (CAUSAL && kj0 + BN - 1 > off) ||
                               (window > 0 && (off + Nq - 1 - kj0 >= window ||
                                               (!CAUSAL && kj0 + BN - 1 - off >= window)));
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          if (4 * (q >> 2) >= Nq) break;  // whole groups of four columns up to Nq
          const int pos = off + q;
          bool vis = q < Nq;
          if (need_mask)
            vis = vis && kj < Nk && (!CAUSAL || kj <= pos) &&
                  (window == 0 || (pos - kj < window && (CAUSAL || kj - pos < window)));
          x[q] = vis ? __uint_as_float(sv[q]) * scale_log2 : -INFINITY;
          // The column's reference max must move: a score beats it by the
          // threshold, or the column sees its first key.
          if (x[q] > m_ref[q] + kDecRescale || (m_ref[q] == -INFINITY && x[q] != -INFINITY)) need |= 1u << q;
        }
        need = __reduce_or_sync(0xffffffffu, need);
      }
      // The warps trade their need bits (buffer j % 2, written again two
      // steps on, after every warp has passed the next step's barrier, by
      // which time all have read it).
      uint32_t* flags = reinterpret_cast<uint32_t*>(red + 3 * 4 * NQ) + b * 4;
      if (lane == 0) flags[warp] = need;
      named_bar_sync(1, 128);
      const uint32_t need_all = flags[0] | flags[1] | flags[2] | flags[3];
      float alpha[NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) alpha[q] = 1.f;
      bool rescale = false;  // the same in every thread: all read the same maxima
      if (need_all != 0) {
        // Some column's reference max moves (the first steps, and rarely
        // after): the column maxima over the step's 128 keys, butterflies per
        // warp in groups of four that interleave, then the four warps through
        // shared memory.  Every warp takes this branch (the bits are common),
        // so the second barrier is met by all of them too.
        if (ok) {
#pragma unroll
          for (int g = 0; g < NQ / 4; ++g) {
            if (4 * g >= Nq) break;
            float v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = x[4 * g + u];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
#pragma unroll
              for (int u = 0; u < 4; ++u) v[u] = fmaxf(v[u], __shfl_xor_sync(0xffffffffu, v[u], o));
            if (lane == 0) {
#pragma unroll
              for (int u = 0; u < 4; ++u) rb[warp * NQ + 4 * g + u] = v[u];
            }
          }
        }
        named_bar_sync(1, 128);
        if (ok) {
#pragma unroll
          for (int q = 0; q < NQ; ++q) {
            if (4 * (q >> 2) >= Nq) break;
            if (!((need_all >> q) & 1u)) continue;
            const float mstep = fmaxf(fmaxf(rb[q], rb[NQ + q]), fmaxf(rb[2 * NQ + q], rb[3 * NQ + q]));
            if (m_ref[q] != -INFINITY) {
              alpha[q] = ex2(m_ref[q] - mstep);
              rescale = true;
            }
            m_ref[q] = mstep;
          }
        }
      }
      if (!ok) continue;
      __half ph[NQ];
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (4 * (q >> 2) >= Nq) break;
        // Weights rounded to f16 as the P V product takes them; the row sums
        // are formed from the rounded values.
        const float p = m_ref[q] == -INFINITY ? 0.f : ex2(x[q] - m_ref[q]);
        ph[q] = __float2half_rn(p);
        lsum[q] = lsum[q] * alpha[q] + __half2float(ph[q]);
      }
      // P^T into buffer b, K-major with 128-byte swizzle: row q (query), key
      // tid in 16-byte granule (tid % 64) / 8 of chunk tid / 64, stored at
      // granule position granule ^ (q % 8).  Rows past Nq are left as they
      // are: they only feed O^T columns that are never read.
      if (j >= 2 && !(ok = mbar_wait_warp(&bars->p_free[b], ((j - 2) >> 1) & 1, wc))) continue;
      {
        uint8_t* pb = smem + C::OFF_P + b * C::P_TILE + (tid >> 6) * C::P_CHUNK;
        const int kc = tid & 63, g = kc >> 3, wb = (kc & 7) * 2;
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          if (4 * (q >> 2) >= Nq) break;
          *reinterpret_cast<__half*>(pb + q * 128 + ((g ^ (q & 7)) << 4) + wb) = ph[q];
        }
      }
      if (rescale) {
        // A column's reference max moved: scale its O^T column (row tid of
        // O^T is this thread's TMEM lane) once the previous P V is done.
        if (j >= 1 && !(ok = mbar_wait_warp(&bars->pv_done, (j - 1) & 1, wc))) continue;
        tc_fence_after();
        uint32_t o[NQ];
        tmem_ld16(tmem + lane_bits + C::TM_O, o);
        tmem_wait_ld();
        reg_fence16(o);
#pragma unroll
        for (int q = 0; q < NQ; ++q)
          if (4 * (q >> 2) < Nq) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha[q]);
        tmem_st16(tmem + lane_bits + C::TM_O, o);
        tmem_wait_st();
      }
      fence_proxy_async_smem();  // P^T to the tensor core
      tc_fence_before();
      mbar_arrive_warp(&bars->p_full[b]);
    }
    // ---------------------------------------------------------- epilogue
    // Column sums over the 128 threads, in a fixed order (the barrier is
    // met by every elementwise warp once).
    float* rs = red + 2 * 4 * NQ;
#pragma unroll
    for (int g = 0; g < NQ / 4; ++g) {
      if (4 * g >= Nq) break;
      float v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = lsum[4 * g + u];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] += __shfl_xor_sync(0xffffffffu, v[u], o);
      if (lane == 0) {
#pragma unroll
        for (int u = 0; u < 4; ++u) rs[warp * NQ + 4 * g + u] = v[u];
      }
    }
    named_bar_sync(1, 128);
    if (ok && ntiles > 0) ok = mbar_wait_warp(&bars->o_full, 0, wc);
    if (ok) {
      uint32_t o[NQ];
      if (ntiles > 0) {
        tc_fence_after();
        tmem_ld16(tmem + lane_bits + C::TM_O, o);
        tmem_wait_ld();
        reg_fence16(o);
      }
      constexpr float kLn2 = 0.6931471805599453f;
#pragma unroll
      for (int q = 0; q < NQ; ++q) {
        if (q >= Nq) break;
        const float l = (rs[q] + rs[NQ + q]) + (rs[2 * NQ + q] + rs[3 * NQ + q]);
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        // Row tid of O^T is column tid of output row q: consecutive threads
        // write consecutive elements.
        const float val = ntiles > 0 ? __uint_as_float(o[q]) * inv_l : 0.f;
        const float L = l > 0.f ? (m_ref[q] + log2f(l)) * kLn2 : -INFINITY;
        if (kv.part_o != nullptr) {
          // Key split: this split's O (normalised within it) and its logsumexp
          // in both slots the merge reads; a query that saw no key here gets
          // O = 0 and -inf.
          const long long prow = (static_cast<long long>(split) * BH + bh) * kv.nq_pad + q;
          if (tid < D) kv.part_o[prow * D + tid] = val;
          if (tid == 0) {
            kv.part_lse[prow] = L;
            kv.part_lseb[prow] = L;
          }
        } else {
          T* orow = out + bb * so.b + hh * so.h + static_cast<long long>(q) * so.n;
          if (tid < D) {
            if constexpr (E::kFmt == 1) orow[tid] = __float2bfloat16_rn(val);
            else orow[tid] = __float2half_rn(val);
          }
          if (tid == 0) lse_out[static_cast<long long>(bh) * Nq + q] = L;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == C::MMA_WARP) tmem_dealloc(tmem, C::TM_COLS);
}

template <typename T, int D, bool CAUSAL>
static cudaError_t launch_decode_t(const FwdArgs& a, cudaStream_t stream) {
  using C = DecCfg<D>;
  auto kern = attn_decode_kernel<T, D, CAUSAL>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), C::SMEM_BYTES, a.device);
  if (e != cudaSuccess) return e;
  if (a.kv.n_splits < 1 || a.N > kDecodeMaxQ || a.kv.nq_pad != C::NQ)
    return note_cuda(cudaErrorInvalidValue, "decode kernel (bad plan)");
  const long long grid = static_cast<long long>(a.BH) * a.kv.n_splits;
  kern<<<static_cast<unsigned>(grid), DecThreads<T>::value, C::SMEM_BYTES, stream>>>(
      *a.tm_q, *a.tm_k, *a.tm_v, static_cast<T*>(a.o), a.so, a.lse, a.N, a.kv.nk, a.H, a.BH, a.window,
      a.scale_log2, a.kv, a.err);
  return note_cuda(cudaGetLastError(), "decode kernel launch");
}

template <typename T>
static cudaError_t launch_decode_dt(const FwdArgs& a, cudaStream_t stream) {
  if (a.d != 128) return note_cuda(cudaErrorInvalidValue, "decode kernel (d = 128 only)");
  return a.causal ? launch_decode_t<T, 128, true>(a, stream) : launch_decode_t<T, 128, false>(a, stream);
}

cudaError_t launch_decode(const FwdArgs& a, cudaStream_t stream) {
  return a.dtype == kF16 ? launch_decode_dt<__half>(a, stream) : launch_decode_dt<__nv_bfloat16>(a, stream);
}

}  // namespace exattn
