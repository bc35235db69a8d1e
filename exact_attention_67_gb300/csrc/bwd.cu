// bwd.cu -- attention backward for sm_103a, recomputing S and P tile by tile
// from the stored logsumexp ("Gemini 3 Flash的注意力内核重写：算子融合如何实现
// 亚毫秒级推理", §4 重计算: keep only the row statistics, recompute the QK^T
// blocks in the backward pass and stream the gradients).  With
// P_ij = exp(scale q_i.k_j - lse_i), dP_ij = dO_i.v_j, D_i = dO_i.O_i and
// dS_ij = P_ij (dP_ij - D_i) (the softmax vector-Jacobian product):
//     dV_j = sum_i P_ij dO_i,  dK_j = scale sum_i dS_ij q_i,  dQ_i = scale sum_j dS_ij k_j.
//
// Three kernels, no atomics (every output element is summed by one CTA in a
// fixed order, so results are bit-identical run to run):
//   1. bwd_rowdot_kernel: D_i = sum_c dO_ic O_ic (bandwidth bound; the
//      separate attn_bwd_preprocess call -- attn_bwd forms D_i inside the
//      dQ kernel).
//   2. bwd_dkdv_kernel: one CTA per 128-key tile; streams query tiles (64
//      queries at d = 128, 96 at d = 64) of Q and dO (TMA ring); per tile
//      the tensor core computes S^T = K Q_i^T and dP^T = V dO_i^T into TMEM,
//      warpgroups (thread = key row; one at d = 128, three at d = 64, each
//      on 32 of the step's query columns) turn them into P^T and dS^T
//      (input type, written back over S^T and dP^T), and the
//      tensor core accumulates dV += P^T dO_i and dK += dS^T Q_i in TMEM.
//      S^T/dP^T are double buffered so the next tile's products overlap the
//      current elementwise work.
//   3. bwd_dq_kernel (dq.cu): two 128-query tiles per CTA; streams key
//      tiles (64 keys at d = 128, 96 at d = 64) of K and V; S = Q K_j^T and
//      dP = dO V_j^T into TMEM, dS (input type) written back, and
//      dQ += dS K_j accumulated in TMEM.  In attn_bwd it runs first and
//      also forms D_i for its rows, which bwd_dkdv_kernel then reads.
// Causal: key tiles wholly above the diagonal are skipped, diagonal tiles are
// masked element by element (key j visible to query i iff j <= i).
#include "kernels.cuh"
#include "ptx.cuh"

namespace exattn {

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------- D_i
template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_rowdot_kernel(const T* __restrict__ o, Strides so,
                                                         const T* __restrict__ dO, Strides sdo,
                                                         const float* __restrict__ o32,
                                                         float* __restrict__ Dout, long long rows, int N, int H,
                                                         bool contiguous) {
  constexpr int TPR = D / 8;  // threads per row, 8 elements (16 bytes) each
  constexpr int RPW = 32 / TPR;
  const int lane = threadIdx.x & 31;
  const long long warp_g = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long n_warps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const int sub = lane / TPR, part = lane % TPR;
  for (long long r0 = warp_g * RPW; r0 < rows; r0 += n_warps * RPW) {
    const long long r = r0 + sub;  // row of [B*H, N]
    float acc = 0.f;
    if (r < rows) {
      const T* orow = o + r * D;
      const T* drow = dO + r * D;
      if (!contiguous) {
        // B*H*N < 2^31 (checked at the C ABI): 32-bit index arithmetic.
        const int ri = static_cast<int>(r), bh = ri / N, n = ri - bh * N, b = bh / H, h = bh - b * H;
        orow = o + b * so.b + h * so.h + n * so.n;
        drow = dO + b * sdo.b + h * sdo.h + n * sdo.n;
      }
      const uint4 c = __ldg(reinterpret_cast<const uint4*>(drow) + part);
      const uint32_t* c2 = reinterpret_cast<const uint32_t*>(&c);
      if (o32 != nullptr) {
        // O in fp32 (contiguous rows): the same 8 elements as two float4.
        const float4* o4 = reinterpret_cast<const float4*>(o32 + r * D) + 2 * part;
        const float4 a0 = __ldg(o4), a1 = __ldg(o4 + 1);
        const float fa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 fc = Elem<T>::unpack(c2[e]);
          acc = fmaf(fa[2 * e], fc.x, acc);
          acc = fmaf(fa[2 * e + 1], fc.y, acc);
        }
      } else {
        const uint4 a = __ldg(reinterpret_cast<const uint4*>(orow) + part);
        const uint32_t* a2 = reinterpret_cast<const uint32_t*>(&a);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 fa = Elem<T>::unpack(a2[e]);
          const float2 fc = Elem<T>::unpack(c2[e]);
          acc = fmaf(fa.x, fc.x, acc);
          acc = fmaf(fa.y, fc.y, acc);
        }
      }
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (r < rows && part == 0) Dout[r] = acc;
  }
}

// ---------------------------------------------------------------- dK, dV
template <int D>
struct DkdvCfg {
  static constexpr int BM = 128;  // keys per CTA (TMEM lanes)
  static constexpr int BR = dkdv_query_step(D);  // queries per step: 64 at d = 128, 96 at d = 64
  static constexpr int NCHUNK = D / 64;
  static constexpr int KCHUNK = BM * 128;  // bytes of one 64-column chunk of a 128-row tile
  static constexpr int QCHUNK = BR * 128;  // ... of a 64-row tile
  static constexpr int KTILE = NCHUNK * KCHUNK;
  static constexpr int QTILE = NCHUNK * QCHUNK;
  static constexpr int STAGES = (D == 64) ? 6 : 4;
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + KTILE;
  static constexpr int OFF_Q = OFF_V + KTILE;
  static constexpr int OFF_DO = OFF_Q + STAGES * QTILE;
  static constexpr int OFF_STAT = OFF_DO + STAGES * QTILE;  // per stage: lse2[BR], D[BR]
  static constexpr int OFF_BAR = OFF_STAT + STAGES * 2 * BR * 4;
  // At least 120 KB so that only one CTA (which holds all 512 TMEM columns) fits on an SM.
  static constexpr int SMEM_BYTES = (OFF_BAR + 512 + 1024 > 120 * 1024) ? OFF_BAR + 512 + 1024 : 120 * 1024;
  static_assert(SMEM_BYTES <= 232448, "over the 227 KB shared-memory limit");
  // Elementwise warps: EW_GROUPS groups of four, one warp per TMEM lane
  // quarter in each group, group g taking query columns BR g / EW_GROUPS
  // onwards of the step.  At d = 64 a step's MMA chain is half as long as at
  // d = 128 while the softmax work is the same, so one group per 32-column
  // chunk (three for the 96-query steps) divides the hand-off latency that
  // bounds it; at d = 128 the chain hides one group's latency and a second
  // costs registers.  Then the producer warp, then the MMA warp.
  static constexpr int QCH = BR / 32;  // 32-column query chunks per step
  static constexpr int EW_GROUPS = D == 64 ? QCH : 1;
  static constexpr int EW_WARPS = 4 * EW_GROUPS;
  static constexpr int PRODUCER_WARP = EW_WARPS, MMA_WARP = EW_WARPS + 1;
  static constexpr int THREADS = 32 * (EW_WARPS + 2);
  // P^T (dS^T) of query chunk ch (32 queries, 16 packed columns) is written
  // from column P_STRIDE ch of S^T (dP^T): with one group a warp owns all of
  // S^T and packs the chunks side by side; with two, each chunk stays inside
  // its own 32 columns, which the other group may not have loaded yet.
  static constexpr int P_STRIDE = EW_GROUPS == 1 ? 16 : 32;
  // Columns of dK / dV read per TMEM round trip in the epilogue (registers
  // for the whole row only with one group).
  static constexpr int EPI_COLS = EW_GROUPS == 1 ? D : 64;
  // Q/dO stage released right after the step's own dV, dK MMAs (d = 64), or
  // inside the next block of score MMAs (d = 128).
  static constexpr bool EARLY_RELEASE = D == 64;
  // TMEM: dK, dV (D columns each), then two buffers of S^T and dP^T (BR
  // columns each): buffer b's S^T at TM_BUF + 2 BR b, its dP^T BR further.
  static constexpr uint32_t TM_DK = 0, TM_DV = D, TM_BUF = 2 * D, TM_COLS = 512;
  static_assert(TM_BUF + 4 * BR <= TM_COLS, "dK, dV and two S^T/dP^T buffers exceed TMEM");
  static_assert(QCH % EW_GROUPS == 0, "each elementwise group takes whole 32-column chunks");
};

template <int STAGES>
struct BwdBars {
  uint64_t kv_full;
  uint64_t st_full[STAGES], st_empty[STAGES];  // streamed operands of one step
  uint64_t s_full[2];                          // both products of buffer b ready
  uint64_t p_full[2];                          // elementwise results of buffer b written
  uint64_t acc_done;
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

template <typename T, int D, bool CAUSAL>
__global__ void __launch_bounds__(DkdvCfg<D>::THREADS, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const float* __restrict__ lse, const float* __restrict__ Dws, T* __restrict__ dk, Strides sdk,
                    T* __restrict__ dv, Strides sdv, int N_max, int H, int BH, int n_ktiles, int group, int window,
                    float scale,
                    float scale_log2, SeqView seq, unsigned* err) {
  using C = DkdvCfg<D>;
  using E = Elem<T>;
  using Bars = BwdBars<C::STAGES>;
  static_assert(sizeof(Bars) <= 512, "barrier block too large");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::OFF_BAR);
  float* stat = reinterpret_cast<float*>(smem + C::OFF_STAT);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  EXATTN_TRACE_INIT();

  // Under the causal mask the first key tiles meet the most queries: run them first.
  const GridPos gp = grid_pos(static_cast<int>(blockIdx.x), BH, n_ktiles, 1, group);
  const int kt = gp.tile;
  const int bh = gp.bh;
  const int hh = bh % H, bb = bh / H;  // head and batch index
  const int k0 = kt * C::BM;
  // This batch's rows (a packed variable-length batch may be shorter than the
  // grid's longest sequence: such a CTA has nothing to do).
  const SeqRows sr0 = seq_rows(seq, bb, hh, H, N_max);
  const int N = sr0.n, row0 = sr0.start, bt = sr0.b_coord;
  if (k0 >= N) return;
  // Queries that see some key of [k0, k0 + BM): from the diagonal (causal) or
  // the window, up to window - 1 past the tile's last key (window W > 0: key j
  // visible to query i iff i - j < W, and also j - i < W without the causal
  // mask).
  const int q_begin = CAUSAL ? k0 : (window > 0 ? max(0, k0 - window + 1) : 0);
  const int q_end = window > 0 ? min(N, min(N, k0 + C::BM) - 1 + window) : N;  // exclusive
  const int i_begin = q_begin / C::BR;
  const int nq = (q_end + C::BR - 1) / C::BR - i_begin;  // >= 1 since k0 < N

  if (threadIdx.x == 0) {
    mbar_init(&bars->kv_full, 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&bars->st_full[s], 1);
      mbar_init(&bars->st_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->p_full[b], 32 * C::EW_WARPS);
    }
    mbar_init(&bars->acc_done, 1);
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
  const uint32_t tmem = bars->tmem_base;
  const WaitCtl wc{&bars->abort, err};

  if (warp == C::PRODUCER_WARP) {
    // ------------------------------------------------------------ producer
    const uint64_t pol_keep = l2_policy_evict_last();  // Q, dO are re-read by every key tile of the head
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(&bars->kv_full, 2 * C::KTILE);
      for (int c = 0; c < C::NCHUNK; ++c) {
        // K, V of this key tile are read by this CTA alone.
        tma_load_4d(&tm_k, &bars->kv_full, smem + C::OFF_K + c * C::KCHUNK, c * 64, row0 + k0, hh, bt,
                    l2_policy_evict_first());
        tma_load_4d(&tm_v, &bars->kv_full, smem + C::OFF_V + c * C::KCHUNK, c * 64, row0 + k0, hh, bt,
                    l2_policy_evict_first());
      }
    }
    // Row terms of the next step are fetched into registers one step ahead, so
    // their global-load latency overlaps the wait for a free stage.
    auto fetch_terms = [&](int it, float (&l2)[C::QCH], float (&dd)[C::QCH]) {
      const int qi0 = (i_begin + it) * C::BR;
#pragma unroll
      for (int u = 0; u < C::QCH; ++u) {
        const int qi = qi0 + lane + 32 * u;
        const bool valid = it < nq && qi < N;
        // Rows past N (zero-filled by TMA) get P = 0 and D = 0: no contribution.
        l2[u] = valid ? lse[sr0.stat0 + qi] * kLog2e : INFINITY;
        dd[u] = valid ? Dws[sr0.stat0 + qi] : 0.f;
      }
    };
    float nl2[C::QCH], ndd[C::QCH];
    fetch_terms(0, nl2, ndd);
    int issued = 0;
    for (int it = 0; it < nq; ++it) {
      const int s = it % C::STAGES;
      const uint32_t ph = (it / C::STAGES) & 1;
      float l2c[C::QCH], ddc[C::QCH];
#pragma unroll
      for (int u = 0; u < C::QCH; ++u) {
        l2c[u] = nl2[u];
        ddc[u] = ndd[u];
      }
      fetch_terms(it + 1, nl2, ndd);
      if (!mbar_wait_warp(&bars->st_empty[s], ph ^ 1, wc)) break;
      if (lane == 0) EXATTN_TRACE_POINT(0, it, 0);
      const int qi0 = (i_begin + it) * C::BR;
      float* st_lse2 = stat + s * 2 * C::BR;
      float* st_D = st_lse2 + C::BR;
      // Stored negated, so the elementwise warps add them.
#pragma unroll
      for (int u = 0; u < C::QCH; ++u) {
        st_lse2[lane + 32 * u] = -l2c[u];
        st_D[lane + 32 * u] = -ddc[u];
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->st_full[s], 2 * C::QTILE);
        for (int c = 0; c < C::NCHUNK; ++c) {
          tma_load_4d(&tm_q, &bars->st_full[s], smem + C::OFF_Q + s * C::QTILE + c * C::QCHUNK, c * 64, row0 + qi0, hh, bt,
                      pol_keep);
          tma_load_4d(&tm_do, &bars->st_full[s], smem + C::OFF_DO + s * C::QTILE + c * C::QCHUNK, c * 64, row0 + qi0, hh, bt,
                      pol_keep);
        }
        EXATTN_TRACE_POINT(0, it, 1);
      }
      issued = it + 1;
    }
    if (lane == 0 && *reinterpret_cast<volatile int*>(&bars->abort)) {
      mbar_wait_drain(&bars->kv_full, 0, err);
      for (int it = max(0, issued - C::STAGES); it < issued; ++it)
        mbar_wait_drain(&bars->st_full[it % C::STAGES], (it / C::STAGES) & 1, err);
    }
    __syncwarp();
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    // Whole-warp loop, elected lane issues (see elect_one()).
    constexpr uint32_t idesc_s = idesc_f16kind(E::kFmt, 128, C::BR, 0, 0);  // K (or V) x Q^T (or dO^T): K-major
    constexpr uint32_t idesc_acc = idesc_f16kind(E::kFmt, 128, D, 0, 1);    // TMEM operand x (Q or dO), MN-major
    const uint64_t k_desc = sdesc_sw128(smem_u32(smem + C::OFF_K), 16, 1024);
    const uint64_t v_desc = sdesc_sw128(smem_u32(smem + C::OFF_V), 16, 1024);
    const uint64_t q_desc = sdesc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
    const uint64_t do_desc = sdesc_sw128(smem_u32(smem + C::OFF_DO), 16, 1024);
    const uint64_t q_mn = sdesc_sw128(smem_u32(smem + C::OFF_Q), C::QCHUNK, 1024);
    const uint64_t do_mn = sdesc_sw128(smem_u32(smem + C::OFF_DO), C::QCHUNK, 1024);
    constexpr uint32_t kQTileDesc = C::QTILE >> 4;
    auto issue_products = [&](int it, int kk0, int kk1) {
      const int s = it % C::STAGES, b = it & 1;
      const uint64_t qa = q_desc + s * kQTileDesc, da = do_desc + s * kQTileDesc;
#pragma unroll
      for (int kk = kk0; kk < kk1; ++kk) {
        const uint32_t ko = ((kk >> 2) * C::KCHUNK + (kk & 3) * 32) >> 4;
        const uint32_t qo = ((kk >> 2) * C::QCHUNK + (kk & 3) * 32) >> 4;
        mma_ss(tmem + C::TM_BUF + b * 2 * C::BR, k_desc + ko, qa + qo, idesc_s, kk > 0);
        mma_ss(tmem + C::TM_BUF + b * 2 * C::BR + C::BR, v_desc + ko, da + qo, idesc_s, kk > 0);
      }
    };
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, wc));
    };
    bool ok = wait_all(&bars->kv_full, 0);
    if (ok) ok = wait_all(&bars->st_full[0], 0);
    if (ok) {
      tc_fence_after();
      if (elect_one()) {
        issue_products(0, 0, D / 16);
        mma_commit(&bars->s_full[0]);
      }
      __syncwarp();
    }
    for (int it = 0; ok && it < nq; ++it) {
      const int s = it % C::STAGES, b = it & 1;
      if (it + 1 < nq) {
        const int s1 = (it + 1) % C::STAGES;
        if (!(ok = wait_all(&bars->st_full[s1], ((it + 1) / C::STAGES) & 1))) break;
        if (lane == 0) EXATTN_TRACE_POINT(1, it, 0);
        tc_fence_after();
        if (elect_one()) {
          // d = 128: the release of step it-1's Q/dO stage rides inside this
          // block (a commit between blocks would hold up the next MMA while
          // the shallow queue in front of the tensor core runs dry); d = 64
          // releases each stage right after its own dV, dK MMAs (below), so
          // that a late stage cannot delay the next release (B4 H32 N4096
          // d64: 1.221 -> 1.201 ms; at d = 128 that order cost 1.7 %).
          issue_products(it + 1, 0, 1);
          if (!C::EARLY_RELEASE && it > 0) mma_commit(&bars->st_empty[(it - 1) % C::STAGES]);
          issue_products(it + 1, 1, D / 16);
          mma_commit(&bars->s_full[b ^ 1]);
        }
        __syncwarp();
        if (lane == 0) EXATTN_TRACE_POINT(1, it, 1);
      }
      if (!(ok = wait_all(&bars->p_full[b], (it >> 1) & 1))) break;
      if (lane == 0) EXATTN_TRACE_POINT(1, it, 2);
      tc_fence_after();
      if (elect_one()) {
        const uint64_t qa = q_mn + s * kQTileDesc, da = do_mn + s * kQTileDesc;
#pragma unroll
        for (int kk = 0; kk < C::BR / 16; ++kk) {
          // dV += P^T dO_i ; dK += dS^T Q_i.  Queries 16 kk .. 16 kk + 15 of
          // P^T (dS^T) sit at column P_STRIDE (kk / 2) + 8 (kk % 2) of S^T (dP^T).
          const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
          const uint32_t col = (kk >> 1) * C::P_STRIDE + (kk & 1) * 8;
          const uint32_t buf = tmem + C::TM_BUF + b * 2 * C::BR;
          mma_ts(tmem + C::TM_DV, buf + col, da + ((kk * 16 * 128) >> 4), idesc_acc, acc);
          mma_ts(tmem + C::TM_DK, buf + C::BR + col, qa + ((kk * 16 * 128) >> 4), idesc_acc, acc);
        }
        if (C::EARLY_RELEASE) {
          mma_commit(&bars->st_empty[s]);
        } else if (it + 1 == nq) {
          if (it > 0) mma_commit(&bars->st_empty[(it - 1) % C::STAGES]);
          mma_commit(&bars->st_empty[s]);
        }
      }
      __syncwarp();
      if (lane == 0) EXATTN_TRACE_POINT(1, it, 3);
    }
    if (elect_one()) {
      if (ok) mma_commit(&bars->acc_done);
      mma_commit(&bars->mma_done);
    }
    __syncwarp();
    if (lane == 0) mbar_wait_drain(&bars->mma_done, 0, err);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ elementwise (thread = key row)
    // Warp w takes TMEM lane quarter w % 4 and the 32-column chunks
    // NC (w / 4) .. NC (w / 4) + NC - 1 of the step's BR query columns.
    constexpr int NC = C::QCH / C::EW_GROUPS;
    const int wq = warp & 3, group = C::EW_GROUPS == 1 ? 0 : warp >> 2;
    const int row = wq * 32 + lane;
    const int key = k0 + row;
    const uint32_t lane_bits = static_cast<uint32_t>(wq * 32) << 16;
    bool ok = true;
    for (int it = 0; ok && it < nq; ++it) {
      const int s = it % C::STAGES, b = it & 1;
      // Per-thread waits on the step's hand-offs (warp-uniform ones cost
      // 1.3 % at d = 64): the lanes enter them converged and see the same
      // barrier phase, abort flag and timer, so they leave them together.
      if (!(ok = mbar_wait(&bars->s_full[b], (it >> 1) & 1, wc))) break;
      if (threadIdx.x == 0) EXATTN_TRACE_POINT(2, it, 0);
      // The row statistics of this step were written by the producer's threads.
      if (!(ok = mbar_wait(&bars->st_full[s], (it / C::STAGES) & 1, wc))) break;
      if (threadIdx.x == 0) EXATTN_TRACE_POINT(2, it, 1);
      tc_fence_after();
      const uint32_t tb = tmem + lane_bits + C::TM_BUF + b * 2 * C::BR;
      uint32_t sr[NC][32], dr[NC][32];
#pragma unroll
      for (int g = 0; g < NC; ++g) {
        tmem_ld32(tb + 32 * (group * NC + g), sr[g]);
        tmem_ld32(tb + C::BR + 32 * (group * NC + g), dr[g]);
      }
      tmem_wait_ld();
#pragma unroll
      for (int g = 0; g < NC; ++g) {
        tmem_reg_fence(sr[g]);
        tmem_reg_fence(dr[g]);
      }
      if (threadIdx.x == 0) EXATTN_TRACE_POINT(2, it, 2);
      const float* st_lse2 = stat + s * 2 * C::BR;
      const float* st_D = st_lse2 + C::BR;
      const int qi0 = (i_begin + it) * C::BR;
      // Some query of this step cannot see some key of the tile: before the
      // diagonal, or outside the window.
      const bool need_mask = (CAUSAL && qi0 < k0 + C::BM) ||
                             (window > 0 && (qi0 + C::BR - 1 - k0 >= window ||
                                             (!CAUSAL && k0 + C::BM - 1 - qi0 >= window)));
      if (need_mask) {
        // Hidden scores become -inf, so P = 0 and dS = 0 there.  Query
        // qi0 + c sees this thread's key iff c lies in [c_lo, c_hi].
        const int c_lo = (CAUSAL ? key : (window > 0 ? key - window + 1 : -C::BR)) - qi0;
        const int c_hi = (window > 0 ? key + window - 1 : qi0 + C::BR) - qi0;
#pragma unroll
        for (int g = 0; g < NC; ++g)
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int c = 32 * (group * NC + g) + e;
            if (c < c_lo || c > c_hi) sr[g][e] = __float_as_uint(-INFINITY);
          }
      }
      // Column statistics come from shared memory as float4 broadcasts: four
      // columns per load keeps the shared-memory pipe free for the TMA and
      // TMEM traffic of the other roles.
      const float4* st_lse4 = reinterpret_cast<const float4*>(st_lse2);
      const float4* st_D4 = reinterpret_cast<const float4*>(st_D);
#pragma unroll
      for (int g = 0; g < NC; ++g) {
        const int ch = group * NC + g;  // chunk of 32 query columns
        uint32_t pk[16], dk_[16];
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const float4 L4 = st_lse4[ch * 8 + q4], D4 = st_D4[ch * 8 + q4];
          const float Lv[4] = {L4.x, L4.y, L4.z, L4.w}, Dv[4] = {D4.x, D4.y, D4.z, D4.w};  // -lse2, -D
          float pv[4], dsv[4];
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int cl = 4 * q4 + w;  // column within the chunk
            pv[w] = ex2(fmaf(__uint_as_float(sr[g][cl]), scale_log2, Lv[w]));
            dsv[w] = pv[w] * (__uint_as_float(dr[g][cl]) + Dv[w]);
          }
          pk[2 * q4] = E::pack(pv[0], pv[1]);
          pk[2 * q4 + 1] = E::pack(pv[2], pv[3]);
          dk_[2 * q4] = E::pack(dsv[0], dsv[1]);
          dk_[2 * q4 + 1] = E::pack(dsv[2], dsv[3]);
        }
        // P^T of queries 32 ch .. 32 ch + 31 at columns P_STRIDE ch onwards,
        // dS^T BR columns further.
        tmem_st16(tb + ch * C::P_STRIDE, pk);
        tmem_st16(tb + C::BR + ch * C::P_STRIDE, dk_);
      }
      tmem_wait_st();
      if (threadIdx.x == 0) EXATTN_TRACE_POINT(2, it, 3);
      tc_fence_before();
      mbar_arrive(&bars->p_full[b]);
    }
    // The first four warps write dK and dV.
    if (ok && group == 0) ok = mbar_wait_warp(&bars->acc_done, 0, wc);
    if (ok && group == 0) {
      tc_fence_after();

      // Rows leave through shared memory (the K, V tiles are no longer read:
      // every MMA is done): each thread writes its row, then each warp stores
      // its 32 rows with coalesced 16-byte lanes (whole rows per instruction)
      // instead of 32 rows 256 bytes apart per instruction.
      constexpr int VPR = D / 8;        // 16-byte vectors per row
      constexpr int RPI = 32 / VPR;     // rows per warp instruction
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t tacc = tmem + lane_bits + (which == 0 ? C::TM_DK : C::TM_DV);
        const float mul = which == 0 ? scale : 1.f;
        const Strides& so = which == 0 ? sdk : sdv;
        uint4* stage = reinterpret_cast<uint4*>(smem + (which == 0 ? C::OFF_K : C::OFF_V)) + warp * 32 * VPR;
        // The row in round trips of EPI_COLS columns to TMEM.
        constexpr int RT = C::EPI_COLS / 32;
#pragma unroll
        for (int c0 = 0; c0 < D / 32; c0 += RT) {
          uint32_t r[RT][32];
#pragma unroll
          for (int cc = 0; cc < RT; ++cc) tmem_ld32(tacc + (c0 + cc) * 32, r[cc]);
          tmem_wait_ld();
#pragma unroll
          for (int cc = 0; cc < RT; ++cc) tmem_reg_fence(r[cc]);
#pragma unroll
          for (int cc = 0; cc < RT; ++cc) {
            const int c = c0 + cc;
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              pk[e] = E::pack(__uint_as_float(r[cc][2 * e]) * mul, __uint_as_float(r[cc][2 * e + 1]) * mul);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)  // vector j of the row at slot j ^ (row % VPR): spreads the banks
              stage[lane * VPR + ((c * 4 + v4) ^ (lane % VPR))] =
                  make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
          }
        }
        __syncwarp();
        T* base = (which == 0 ? dk : dv) + bt * so.b + hh * so.h;
#pragma unroll
        for (int i = 0; i < VPR; ++i) {
          const int rl = i * RPI + lane / VPR, j = lane % VPR;  // row within the warp, vector within the row
          const int krow = k0 + warp * 32 + rl;
          if (krow < N)
            reinterpret_cast<uint4*>(base + static_cast<long long>(row0 + krow) * so.n)[j] =
                stage[rl * VPR + (j ^ (rl % VPR))];
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == C::MMA_WARP) tmem_dealloc(tmem, C::TM_COLS);
}

// ---------------------------------------------------------------- launch
template <typename T, int D>
static cudaError_t launch_prep_t(const BwdArgs& a, cudaStream_t stream) {
  // Packed variable-length sequences are one batch of `total` rows per head.
  const int n_rows = a.seq.cu_seqlens ? a.seq.total : a.N;
  const long long rows = static_cast<long long>(a.seq.cu_seqlens ? a.H : a.BH) * n_rows;
  const int rpb = 256 / (D / 8);  // rows per 256-thread block
  long long blocks = (rows + rpb - 1) / rpb;
  if (blocks > 152 * 16) blocks = 152 * 16;
  // "contiguous": O and dO both [B, H, N, d] packed (O unused when the fp32
  // copy o32, always packed, replaces it).
  const Strides& so = a.o32 ? a.sdo : a.so;
  bwd_rowdot_kernel<T, D><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      static_cast<const T*>(a.o), a.so, static_cast<const T*>(a.dO), a.sdo, a.o32, a.D, rows, n_rows, a.H,
      so.n == D && so.h == static_cast<long long>(n_rows) * D && so.b == static_cast<long long>(a.H) * n_rows * D &&
          a.sdo.n == so.n && a.sdo.h == so.h && a.sdo.b == so.b);
  return note_cuda(cudaGetLastError(), "row-dot kernel launch");
}

template <typename T, int D, bool CAUSAL>
static cudaError_t launch_dkdv_t(const BwdArgs& a, cudaStream_t stream) {
  using C = DkdvCfg<D>;
  auto kern = bwd_dkdv_kernel<T, D, CAUSAL>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), C::SMEM_BYTES, a.device);
  if (e != cudaSuccess) return e;
  const int n_kt = (a.N + C::BM - 1) / C::BM;
  // Q, dO of a group's problems stay in a quarter of L2: every key-tile CTA
  // of a problem re-reads them over the group's waves (B4 H32 N4096 d64:
  // 1.323 ms with half of L2, 1.280 ms with a quarter; B1 H16 N8192 and B1 H8
  // N16384 d128 unchanged within 0.5 %).
  const int group = l2_group(2ll * a.N * D * static_cast<long long>(sizeof(T)), a.BH, kL2GroupBytes / 2);
  kern<<<static_cast<unsigned>(static_cast<long long>(n_kt) * a.BH), C::THREADS, C::SMEM_BYTES, stream>>>(
      *a.tm_qkv, *a.tm_k128, *a.tm_v128, *a.tm_dokv, a.lse, a.D, static_cast<T*>(a.dk), a.sdk,
      static_cast<T*>(a.dv), a.sdv, a.N, a.H, a.BH, n_kt, group, a.window, a.scale, a.scale_log2, a.seq, a.err);
  return note_cuda(cudaGetLastError(), "dK/dV kernel launch");
}

template <typename T>
static cudaError_t launch_prep_dt(const BwdArgs& a, cudaStream_t stream) {
  return a.d == 64 ? launch_prep_t<T, 64>(a, stream) : launch_prep_t<T, 128>(a, stream);
}

template <typename T>
static cudaError_t launch_dkdv_dt(const BwdArgs& a, cudaStream_t stream) {
  if (a.d == 64) return a.causal ? launch_dkdv_t<T, 64, true>(a, stream) : launch_dkdv_t<T, 64, false>(a, stream);
  return a.causal ? launch_dkdv_t<T, 128, true>(a, stream) : launch_dkdv_t<T, 128, false>(a, stream);
}

cudaError_t launch_bwd_prep(const BwdArgs& a, cudaStream_t stream) {
  return a.dtype == kF16 ? launch_prep_dt<__half>(a, stream) : launch_prep_dt<__nv_bfloat16>(a, stream);
}

cudaError_t launch_bwd_dkdv(const BwdArgs& a, cudaStream_t stream) {
  return a.dtype == kF16 ? launch_dkdv_dt<__half>(a, stream) : launch_dkdv_dt<__nv_bfloat16>(a, stream);
}

}  // namespace exattn
