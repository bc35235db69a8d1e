// dq.cu -- the dQ part of the attention backward for sm_103a, atomic-free.
//
// dQ_i = scale sum_j dS_ij k_j with dS_ij = P_ij (dP_ij - D_i), P_ij =
// exp(scale q_i.k_j - lse_i) recomputed tile by tile from the stored
// logsumexp ("Gemini 3 Flash的注意力内核重写：算子融合如何实现亚毫秒级推理",
// §4 重计算).  Every dQ row is summed by one CTA in a fixed key order, so the
// result is bit-identical run to run without atomics.
//
// GB300 mapping (one CTA per SM, 352 threads), the same ping-pong as the
// forward kernel:
//   * the CTA owns two 128-row query tiles of one (batch, head); Q and dO of
//     both stay in shared memory, key tiles of K and V (64 keys at d = 128,
//     96 at d = 64) stream through a TMA ring that both query tiles share;
//   * warp 9 + t issues the MMAs of query tile t (warp-uniform loop, elected
//     lane): per key step, dQ_t += dS_t K_j with dS_t read from TMEM, then
//     S_t = Q_t K_j+1^T and dP_t = dO_t V_j+1^T into TMEM.  With one issuer
//     per tile the tensor core always has queued work while the other issuer
//     waits on its tile's hand-off;
//   * warps 0-3 / 4-7 turn S_t, dP_t into dS_t (input type, written over S_t) for
//     tile 0 / tile 1 (thread = query row); while one warpgroup works, the
//     tensor core runs the other tile's MMAs, which hides the hand-off
//     latency between the two roles;
//   * warp 8 issues the TMA loads;
//   * when the kernel forms the row terms (attn_bwd), warps 0-7 first compute
//     D_i = dO_i . O_i for their rows, O read from global memory and dO from
//     its tile in shared memory, with the separate row-dot kernel's lane
//     grouping and summation order (bit-identical D), and store D for the
//     dK/dV kernel that runs next.
// TMEM per tile t (base 256 t): d = 128: dQ_t [0,128), S_t [128,192), dP_t
// [192,256); d = 64: dQ_t [0,64), S_t [64,160), dP_t [160,256).
// Causal: key tiles above the diagonal are skipped per query tile, diagonal
// tiles masked per element (key j visible to query i iff j <= i).
#include "kernels.cuh"
#include "ptx.cuh"

namespace exattn {

namespace {

constexpr float kLog2eDq = 1.4426950408889634f;

template <int D>
struct DqCfg {
  static constexpr int BM = 128;  // queries per tile (TMEM lanes); two tiles per CTA
  static constexpr int BN = dq_key_step(D);  // keys per step: 64 at d = 128, 96 at d = 64
  static constexpr int NCHUNK = D / 64;
  static constexpr int QCHUNK = BM * 128;
  static constexpr int KCHUNK = BN * 128;
  static constexpr int QTILE = NCHUNK * QCHUNK;
  static constexpr int KTILE = NCHUNK * KCHUNK;
  static constexpr int STAGES = (D == 64) ? 6 : 3;
  static constexpr int OFF_Q = 0;                      // Q_0, Q_1
  static constexpr int OFF_DO = OFF_Q + 2 * QTILE;     // dO_0, dO_1
  static constexpr int OFF_K = OFF_DO + 2 * QTILE;
  static constexpr int OFF_V = OFF_K + STAGES * KTILE;
  static constexpr int OFF_BAR = OFF_V + STAGES * KTILE;
  static constexpr int SMEM_BYTES = (OFF_BAR + 512 + 1024 > 120 * 1024) ? OFF_BAR + 512 + 1024 : 120 * 1024;
  static_assert(SMEM_BYTES <= 232448, "over the 227 KB shared-memory limit");
  static constexpr int THREADS = 352;  // warps 0-7 elementwise (two tiles), 8 producer, 9-10 MMA
  // TMEM per tile t (base 256 t): dQ_t, then S_t and dP_t of BN columns each.
  static constexpr uint32_t TM_TILE = 256, TM_DQ = 0, TM_S = D == 64 ? 64 : 128, TM_DP = TM_S + BN, TM_COLS = 512;
  static_assert(TM_DQ + D <= TM_S && TM_DP + BN <= TM_TILE, "a tile's dQ, S, dP exceed its 256 TMEM columns");
  static_assert(BN == 64 || BN == 96, "the elementwise step handles two or three 32-column chunks");
};

template <int STAGES>
struct DqBars {
  uint64_t qd_full[2];                         // Q_t and dO_t loaded
  uint64_t st_full[STAGES], st_empty[STAGES];  // K_j, V_j
  uint64_t s_full[2];                          // S_t, dP_t ready
  uint64_t p_full[2];                          // dS_t written by the 128 threads of tile t
  uint64_t acc_done[2];                        // dQ_t final
  uint64_t turn[2];                            // issuer t may queue its next block of MMAs
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

}  // namespace

template <typename T, int D, bool CAUSAL>
__global__ void __launch_bounds__(DqCfg<D>::THREADS, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const float* __restrict__ lse, float* __restrict__ Dws, const T* __restrict__ o, Strides so,
                  const T* __restrict__ dO, Strides sdo, const float* __restrict__ o32, T* __restrict__ dq,
                  Strides sdq, int N_max, int H, int BH, int n_pairs, int group, int window, float scale,
                  float scale_log2, SeqView seq, unsigned* err) {
  using C = DqCfg<D>;
  using E = Elem<T>;
  using Bars = DqBars<C::STAGES>;
  static_assert(sizeof(Bars) <= 512, "barrier block too large");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::OFF_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  EXATTN_TRACE_INIT();

  // Under the causal mask the last query tiles meet the most keys: run them first.
  const GridPos gp = grid_pos(static_cast<int>(blockIdx.x), BH, n_pairs, 1, group);
  const int pair = n_pairs - 1 - gp.tile;
  const int bh = gp.bh;
  const int hh = bh % H, bb = bh / H;  // head and batch index
  const int q0 = pair * 2 * C::BM;
  // This batch's rows (a packed variable-length batch may be shorter than the
  // grid's longest sequence: such a CTA has nothing to do).
  const SeqRows sr0 = seq_rows(seq, bb, hh, H, N_max);
  const int N = sr0.n, row0 = sr0.start, bt = sr0.b_coord;
  if (q0 >= N) return;
  // Keys any row of query tile t can see (as in the forward): up to the
  // diagonal or window - 1 past its last row, from the window start of the
  // pair's first row; both tiles stream key steps from kv_lo.
  auto key_end = [&](int t) {  // exclusive
    const int r0 = q0 + t * C::BM, r1 = min(N, r0 + C::BM);
    if (r0 >= N) return 0;
    if (CAUSAL) return r1;
    return window > 0 ? min(N, r1 - 1 + window) : N;
  };
  const int kv_lo = window > 0 ? max(0, q0 - window + 1) / C::BN : 0;
  // Key steps of query tile t, counted from kv_lo (0 if the tile lies wholly past N).
  auto steps_for = [&](int t) {
    const int e = key_end(t);
    return e == 0 ? 0 : (e + C::BN - 1) / C::BN - kv_lo;
  };
  const int nk0 = steps_for(0), nk1 = steps_for(1);
  const int n_iter = max(nk0, nk1);

  if (threadIdx.x == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->qd_full[t], 1);
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 128);
      mbar_init(&bars->acc_done[t], 1);
      mbar_init(&bars->turn[t], 1);
    }
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&bars->st_full[s], 1);
      mbar_init(&bars->st_empty[s], 2);  // one commit (or arrive) per query tile
    }
    mbar_init(&bars->mma_done, 2);
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
      const uint64_t pol_keep = l2_policy_evict_last();  // K, V are re-read by every query pair of the head
      const uint64_t pol_once = l2_policy_evict_first();
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if ((t == 0 ? nk0 : nk1) == 0) continue;
        mbar_arrive_expect_tx(&bars->qd_full[t], 2 * C::QTILE);
        for (int c = 0; c < C::NCHUNK; ++c) {
          tma_load_4d(&tm_q, &bars->qd_full[t], smem + C::OFF_Q + t * C::QTILE + c * C::QCHUNK, c * 64,
                      row0 + q0 + t * C::BM, hh, bt, pol_once);
          tma_load_4d(&tm_do, &bars->qd_full[t], smem + C::OFF_DO + t * C::QTILE + c * C::QCHUNK, c * 64,
                      row0 + q0 + t * C::BM, hh, bt, pol_once);
        }
      }
      int issued = 0;
      for (int it = 0; it < n_iter; ++it) {
        const int s = it % C::STAGES;
        const uint32_t ph = (it / C::STAGES) & 1;
        if (!mbar_wait(&bars->st_empty[s], ph ^ 1, wc)) break;
        EXATTN_TRACE_POINT(0, it, 0);
        mbar_arrive_expect_tx(&bars->st_full[s], 2 * C::KTILE);
        for (int c = 0; c < C::NCHUNK; ++c) {
          tma_load_4d(&tm_k, &bars->st_full[s], smem + C::OFF_K + s * C::KTILE + c * C::KCHUNK, c * 64,
                      row0 + (kv_lo + it) * C::BN, hh, bt, pol_keep);
          tma_load_4d(&tm_v, &bars->st_full[s], smem + C::OFF_V + s * C::KTILE + c * C::KCHUNK, c * 64,
                      row0 + (kv_lo + it) * C::BN, hh, bt, pol_keep);
        }
        issued = it + 1;
      }
      if (*reinterpret_cast<volatile int*>(&bars->abort)) {
        // Never leave a copy in flight into shared memory this CTA is about to release.
        for (int t = 0; t < 2; ++t)
          if ((t == 0 ? nk0 : nk1) > 0) mbar_wait_drain(&bars->qd_full[t], 0, err);
        for (int it = max(0, issued - C::STAGES); it < issued; ++it)
          mbar_wait_drain(&bars->st_full[it % C::STAGES], (it / C::STAGES) & 1, err);
      }
    }
    __syncwarp();
  } else if (warp >= 9) {
    // ------------------------------------------------------------ MMA issuers: warp 9 + t drives query tile t
    // (whole warp, elected lane issues).  Two issuers keep the tensor core fed
    // while either one waits on its tile's elementwise warps.
    const int t = warp - 9;
    const int nk_t = t == 0 ? nk0 : nk1;
    constexpr uint32_t idesc_s = idesc_f16kind(E::kFmt, 128, C::BN, 0, 0);  // Q (dO) x K^T (V^T): both K-major
    constexpr uint32_t idesc_acc = idesc_f16kind(E::kFmt, 128, D, 0, 1);    // dS from TMEM x K (MN-major)
    const uint64_t q_desc = sdesc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
    const uint64_t do_desc = sdesc_sw128(smem_u32(smem + C::OFF_DO), 16, 1024);
    const uint64_t k_desc = sdesc_sw128(smem_u32(smem + C::OFF_K), 16, 1024);
    const uint64_t v_desc = sdesc_sw128(smem_u32(smem + C::OFF_V), 16, 1024);
    const uint64_t k_mn = sdesc_sw128(smem_u32(smem + C::OFF_K), C::KCHUNK, 1024);
    constexpr uint32_t kQTileDesc = C::QTILE >> 4, kKTileDesc = C::KTILE >> 4;

    auto issue_products = [&](int t, int stage, int kk0, int kk1) {
      const uint32_t base = tmem + t * C::TM_TILE;
      const uint64_t qa = q_desc + t * kQTileDesc, da = do_desc + t * kQTileDesc;
      const uint64_t ka = k_desc + stage * kKTileDesc, va = v_desc + stage * kKTileDesc;
#pragma unroll
      for (int kk = kk0; kk < kk1; ++kk) {
        const uint32_t qo = ((kk >> 2) * C::QCHUNK + (kk & 3) * 32) >> 4;
        const uint32_t ko = ((kk >> 2) * C::KCHUNK + (kk & 3) * 32) >> 4;
        mma_ss(base + C::TM_S, qa + qo, ka + ko, idesc_s, kk > 0);
        mma_ss(base + C::TM_DP, da + qo, va + ko, idesc_s, kk > 0);
      }
    };
    auto issue_dq = [&](int t, int stage, bool acc) {
      const uint32_t base = tmem + t * C::TM_TILE;
      const uint64_t ka = k_mn + stage * kKTileDesc;
#pragma unroll
      for (int kk = 0; kk < C::BN / 16; ++kk)
        mma_ts(base + C::TM_DQ, base + C::TM_S + kk * 8, ka + ((kk * 16 * 128) >> 4), idesc_acc,
               (acc || kk > 0) ? 1u : 0u);
    };
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, wc));
    };

    bool ok = true;
    if (nk_t > 0) {
      ok = wait_all(&bars->qd_full[t], 0) && wait_all(&bars->st_full[0], 0);
      if (ok) {
        tc_fence_after();
        if (elect_one()) {
          issue_products(t, 0, 0, D / 16);
          mma_commit(&bars->s_full[t]);
        }
        __syncwarp();
      }
    }
    // The two issuers take turns, one block of MMAs (dQ_t, then the next S_t,
    // dP_t) each, and pass the turn once their block is issued: the other
    // issuer, already past its own waits, queues its block right behind.
    // (Passing the turn a few MMAs before the end of the block measured
    // slower: two k-steps early cost dQ 7 % at d = 128, one 4 % at d = 64;
    // committing S_t's barrier before passing the turn, not after, gains 1 %.)
    for (int it = 0; ok && it < n_iter; ++it) {
      const int s = it % C::STAGES;
      const uint32_t turn_par = static_cast<uint32_t>(it & 1) ^ (t == 0 ? 1u : 0u);
      if (it >= nk_t) {
        // No MMA of this tile reads stage s: release it once it holds step it's K, V.
        if (!(ok = wait_all(&bars->st_full[s], (it / C::STAGES) & 1))) break;
        if (lane == 0) mbar_arrive(&bars->st_empty[s]);
        if (!(ok = wait_all(&bars->turn[t], turn_par))) break;
        if (lane == 0) mbar_arrive(&bars->turn[t ^ 1]);
        __syncwarp();
        continue;
      }
      const bool more = it + 1 < nk_t;
      const int s1 = (it + 1) % C::STAGES;
      if (!(ok = wait_all(&bars->p_full[t], it & 1))) break;
      if (more && !(ok = wait_all(&bars->st_full[s1], ((it + 1) / C::STAGES) & 1))) break;
      if (!(ok = wait_all(&bars->turn[t], turn_par))) break;
      if (lane == 0) EXATTN_TRACE_POINT(1, it, 4 * t + 0);
      tc_fence_after();
      if (elect_one()) {
        issue_dq(t, s, it > 0);
        mma_commit(&bars->st_empty[s]);  // this tile's last read of K_it, V_it
        if (more) {
          // S_t, dP_t of the next step overwrite the dS_t the dQ MMA just read:
          // the tensor core runs one thread's MMAs in issue order.
          issue_products(t, s1, 0, D / 16);
          mma_commit(&bars->s_full[t]);
          mbar_arrive(&bars->turn[t ^ 1]);
        } else {
          mbar_arrive(&bars->turn[t ^ 1]);
          mma_commit(&bars->acc_done[t]);
        }
      }
      __syncwarp();
      if (lane == 0) EXATTN_TRACE_POINT(1, it, 4 * t + 1);
    }
    if (elect_one()) mma_commit(&bars->mma_done);
    __syncwarp();
    if (lane == 0) mbar_wait_drain(&bars->mma_done, 0, err);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ elementwise (thread = query row of tile t)
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const int tile_r0 = q0 + t * C::BM;
    const int qrow = tile_r0 + row;
    const int nk_t = t == 0 ? nk0 : nk1;
    const uint32_t lane_bits = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tbase = tmem + lane_bits + t * C::TM_TILE;
    const bool valid = qrow < N;
    // Rows past N (zero-filled by TMA) get P = 0 and D = 0: no contribution.
    const float neg_lse2 = valid ? -lse[sr0.stat0 + qrow] * kLog2eDq : -INFINITY;
    bool ok = nk_t > 0;
    float Drow = 0.f;
    if (ok && (o != nullptr || o32 != nullptr)) {
      // D_i = sum_c dO_ic O_ic of the warp's 32 rows, computed here and
      // stored for the dK/dV kernel that runs next.  TPR lanes share a row,
      // 8 columns (one 16-byte granule) each, in the row-dot kernel's
      // grouping and order (each lane's 8 products chained by fma from 0,
      // then a butterfly over the row's lanes), so D is bit-identical to that
      // kernel's.  A lane's O granules are all requested before the wait for
      // Q_t, dO_t; dO is then read from its 128-byte-swizzled tile in shared
      // memory (granule g of row r at g ^ (r mod 8)).
      constexpr int TPR = D / 8, RPW = 32 / TPR, NI = 32 / RPW;
      const int sub = lane / TPR, part = lane % TPR;
      const int pc = part >> 3, pg = part & 7;  // 64-column chunk, granule within it
      const uint8_t* do_tile = smem + C::OFF_DO + t * C::QTILE + pc * C::QCHUNK;
      // Sum over the row's lanes; row i * RPW + s of the warp's 32 belongs to
      // lane i * RPW + s and its sum sits in lanes s * TPR ... s * TPR + TPR - 1.
      auto finish = [&](int i, float a) {
#pragma unroll
        for (int off = TPR / 2; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
#pragma unroll
        for (int s2 = 0; s2 < RPW; ++s2) {
          const float v = __shfl_sync(0xffffffffu, a, s2 * TPR);
          if (lane == i * RPW + s2) Drow = v;
        }
      };
      if (o32 == nullptr) {
        float acc[NI];
        uint4 oa[NI];
#pragma unroll
        for (int i = 0; i < NI; ++i) {
          const int rr = tile_r0 + wq * 32 + i * RPW + sub;
          oa[i] = rr < N ? __ldg(reinterpret_cast<const uint4*>(
                               o + bt * so.b + hh * so.h + static_cast<long long>(row0 + rr) * so.n) + part)
                         : make_uint4(0u, 0u, 0u, 0u);
        }
        ok = mbar_wait_warp(&bars->qd_full[t], 0, wc);
#pragma unroll
        for (int i = 0; i < NI; ++i) {
          const int r = wq * 32 + i * RPW + sub;  // row within the tile
          acc[i] = 0.f;
          if (ok && tile_r0 + r < N) {
            const uint4 c = *reinterpret_cast<const uint4*>(do_tile + r * 128 + ((pg ^ (r & 7)) << 4));
            const uint32_t* a2 = reinterpret_cast<const uint32_t*>(&oa[i]);
            const uint32_t* c2 = reinterpret_cast<const uint32_t*>(&c);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 fa = E::unpack(a2[e]);
              const float2 fc = E::unpack(c2[e]);
              acc[i] = fmaf(fa.x, fc.x, acc[i]);
              acc[i] = fmaf(fa.y, fc.y, acc[i]);
            }
          }
        }
#pragma unroll
        for (int i = 0; i < NI; ++i) finish(i, acc[i]);
      } else {
        // fp32 O, contiguous [B*H, N, d] rows (fixed-length calls only).
        ok = mbar_wait_warp(&bars->qd_full[t], 0, wc);
#pragma unroll 4
        for (int i = 0; i < NI; ++i) {
          const int r = wq * 32 + i * RPW + sub;
          float acc = 0.f;
          if (ok && tile_r0 + r < N) {
            const float4* o4 =
                reinterpret_cast<const float4*>(o32 + (static_cast<long long>(bh) * N + tile_r0 + r) * D) + 2 * part;
            const float4 a0 = __ldg(o4), a1 = __ldg(o4 + 1);
            const float fa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const uint4 c = *reinterpret_cast<const uint4*>(do_tile + r * 128 + ((pg ^ (r & 7)) << 4));
            const uint32_t* c2 = reinterpret_cast<const uint32_t*>(&c);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 fc = E::unpack(c2[e]);
              acc = fmaf(fa[2 * e], fc.x, acc);
              acc = fmaf(fa[2 * e + 1], fc.y, acc);
            }
          }
          finish(i, acc);
        }
      }
      if (ok && valid) Dws[sr0.stat0 + qrow] = Drow;
    } else if (valid) {
      Drow = Dws[sr0.stat0 + qrow];
    }
    for (int it = 0; ok && it < nk_t; ++it) {
      // Per-thread wait on the step's hand-off (a warp-uniform one cost dQ
      // 1.5 %): the lanes enter it converged and see the same barrier phase,
      // abort flag and timer, so they leave it together.
      if (!(ok = mbar_wait(&bars->s_full[t], it & 1, wc))) break;
      if (row == 0) EXATTN_TRACE_POINT(2 + t, it, 0);
      tc_fence_after();
      uint32_t sa[32], da[32], sb[32], db[32];
      tmem_ld32(tbase + C::TM_S, sa);
      tmem_ld32(tbase + C::TM_S + 32, sb);
      tmem_ld32(tbase + C::TM_DP, da);
      tmem_ld32(tbase + C::TM_DP + 32, db);
      tmem_wait_ld();
      tmem_reg_fence(sa);
      tmem_reg_fence(sb);
      tmem_reg_fence(da);
      tmem_reg_fence(db);
      const int kj0 = (kv_lo + it) * C::BN;
      const bool need_mask = (CAUSAL && kj0 + C::BN - 1 > tile_r0) || (kj0 + C::BN > N) ||
                             (window > 0 && (kj0 < tile_r0 + C::BM - window ||
                                             (!CAUSAL && kj0 + C::BN - 1 > tile_r0 + window - 1)));
      // Hidden scores become -inf, so P = 0 and dS = 0 there: key column c
      // is visible to this row iff lo <= c < lim.
      int lim = C::BN, lo = 0;
      if (need_mask) {
        lim = N - kj0;
        if (CAUSAL) lim = min(lim, qrow - kj0 + 1);
        else if (window > 0) lim = min(lim, qrow + window - kj0);
        lo = window > 0 ? qrow - window + 1 - kj0 : 0;
      }
      const float2 sc2 = make_float2(scale_log2, scale_log2), nl2 = make_float2(neg_lse2, neg_lse2);
      const float2 nD2 = make_float2(-Drow, -Drow);
      auto mask = [&](int h, uint32_t (&sv)[32]) {
        if (need_mask) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (h * 32 + e >= lim || h * 32 + e < lo) sv[e] = __float_as_uint(-INFINITY);
        }
      };
      // dS of 32 key columns (chunk h of S and dP, in registers), written as
      // 16 packed columns over the first half of S: chunk h's output lands on
      // columns of chunks already read.
      auto chunk = [&](int h, const uint32_t (&sv)[32], const uint32_t (&dv)[32]) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          // Packed fp32 pairs: one instruction per two columns.
          const float2 y = ffma2(make_float2(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), sc2, nl2);
          const float2 p = make_float2(ex2(y.x), ex2(y.y));
          const float2 dsv =
              fmul2(p, fadd2(make_float2(__uint_as_float(dv[2 * e]), __uint_as_float(dv[2 * e + 1])), nD2));
          pk[e] = E::pack(dsv.x, dsv.y);
        }
        tmem_st16(tbase + C::TM_S + h * 16, pk);
      };
      mask(0, sa);
      mask(1, sb);
      chunk(0, sa, da);
      if constexpr (C::BN == 96) {
        // A third chunk, loaded into chunk 0's registers once those are
        // consumed, under chunk 1's math.
        tmem_ld32(tbase + C::TM_S + 64, sa);
        tmem_ld32(tbase + C::TM_DP + 64, da);
      }
      chunk(1, sb, db);
      if constexpr (C::BN == 96) {
        tmem_wait_ld();
        tmem_reg_fence(sa);
        tmem_reg_fence(da);
        mask(2, sa);
        chunk(2, sa, da);
      }
      tmem_wait_st();
      if (lane == 0) EXATTN_TRACE_POINT(2 + t, it, 1 + wq);
      tc_fence_before();
      mbar_arrive(&bars->p_full[t]);
    }
    if (ok && nk_t > 0) ok = mbar_wait_warp(&bars->acc_done[t], 0, wc);
    if (ok && nk_t > 0) {
      tc_fence_after();
      T* dst_row = dq + bt * sdq.b + hh * sdq.h + static_cast<long long>(row0 + qrow) * sdq.n;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tbase + C::TM_DQ + c * 32, r);
        tmem_wait_ld();
        tmem_reg_fence(r);
        if (valid) {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = E::pack(__uint_as_float(r[2 * e]) * scale, __uint_as_float(r[2 * e + 1]) * scale);
          uint4* dst = reinterpret_cast<uint4*>(dst_row + c * 32);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4)
            dst[v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, C::TM_COLS);
}

template <typename T, int D, bool CAUSAL>
static cudaError_t launch_dq_t(const BwdArgs& a, cudaStream_t stream) {
  using C = DqCfg<D>;
  auto kern = bwd_dq_kernel<T, D, CAUSAL>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), C::SMEM_BYTES, a.device);
  if (e != cudaSuccess) return e;
  const int n_pairs = (a.N + 2 * C::BM - 1) / (2 * C::BM);
  // K, V of a group's heads fill a quarter of L2 (B4 H32 N4096 d64: 612-743 MB
  // per launch with half of L2, 327 MB with a quarter; 339.7 MB algorithmic).
  const int group = l2_group(2ll * a.N * D * static_cast<long long>(sizeof(T)), a.BH, kL2GroupBytes / 2);
  // With a.dq_computes_D the kernel forms D_i from O (or the fp32 copy) and
  // dO and writes it to a.D; otherwise it reads a.D.
  const T* o = a.dq_computes_D ? static_cast<const T*>(a.o) : nullptr;
  const float* o32 = a.dq_computes_D ? a.o32 : nullptr;
  kern<<<static_cast<unsigned>(static_cast<long long>(n_pairs) * a.BH), C::THREADS, C::SMEM_BYTES, stream>>>(
      *a.tm_q128, *a.tm_kdq, *a.tm_vdq, *a.tm_do128, a.lse, a.D, o, a.so, static_cast<const T*>(a.dO), a.sdo, o32,
      static_cast<T*>(a.dq), a.sdq, a.N, a.H, a.BH, n_pairs, group, a.window, a.scale, a.scale_log2, a.seq, a.err);
  return note_cuda(cudaGetLastError(), "dQ kernel launch");
}

template <typename T>
static cudaError_t launch_dq_dt(const BwdArgs& a, cudaStream_t stream) {
  if (a.d == 64) return a.causal ? launch_dq_t<T, 64, true>(a, stream) : launch_dq_t<T, 64, false>(a, stream);
  return a.causal ? launch_dq_t<T, 128, true>(a, stream) : launch_dq_t<T, 128, false>(a, stream);
}

cudaError_t launch_bwd_dq(const BwdArgs& a, cudaStream_t stream) {
  return a.dtype == kF16 ? launch_dq_dt<__half>(a, stream) : launch_dq_dt<__nv_bfloat16>(a, stream);
}

}  // namespace exattn
