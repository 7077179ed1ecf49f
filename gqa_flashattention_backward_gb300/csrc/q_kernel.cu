// Query-stationary tcgen05 kernels: one CTA owns 128 query rows of one query
// head and streams the 64-row key/value tiles it can see.
//
//   FWD : forward with causal / sliding-window / attention-sink masking
//         (tilelang-ascend PR #1638 "Add GQA Sink Backward BHSD", 4->2 commit:
//         "flashattn_fwd: online softmax + sink + window -> O, lse").  Two passes
//         over the key tiles: the first finds each row's maximum logit (sink
//         included; no exponentials), the second forms P = exp(S - max) <= 1 and
//         accumulates P.[V | 1] in TMEM, whose extra column is the row sum l, so
//         O = (P.V) / l and LSE = max + log l with no rescaling of O (head dim
//         128: P.V, with l added up in fp32 by the softmax warpgroups).
//   DQ  : the query-stationary dQ pass (deterministic mode, and the dQ of head
//         dim 192): S = Q.K^T, dP = dO.V^T, dS = P*(dP - Delta) (same PR, review
//         thread k1..k5, in the loop order the Ascend kernel uses for dQ,
//         "dQ[L0C accumulate]"); dQ = scale * dS.K accumulates in TMEM with no
//         atomics.
//
// Warp roles (320 threads): warps 0-3 and 4-7 are two softmax warpgroups that
// take alternate key tiles (warpgroup w the tiles with index parity w), thread r
// owns query row r = TMEM lane r; warp 8 = TMA producer; warp 9 = TMEM allocator
// + MMA issuer (the whole warp runs the loop, one lane elected per MMA).  Tile
// `it` has the TMEM buffer it % NBUF: while one warpgroup works on its tile the
// tensor core computes the other's; with four buffers (the forward of head dim
// 192) it also computes each warpgroup's next tile ahead.  The forward of head
// dims 64 and 128 runs two CTAs per SM, whose warps fill each other's waits.  Operands live in shared memory in the 128-byte
// swizzled layout TMA writes; S, dP, O, dQ accumulate in TMEM; P / dS are packed
// to 16 bits in TMEM and feed the next MMA as its A operand.
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <type_traits>
#include "common.cuh"
#include "umma.cuh"
#include "launch.h"

namespace gqa {

template <int DQK, int DV, bool FWD>
struct QCfg {
  static constexpr int BQ = 128;  // query rows = TMEM lanes
  static constexpr int BK = 64;   // keys per tile
  static constexpr int QB = DQK / 64, VB = DV / 64;  // 64-column (128-byte) blocks
  static constexpr int Q_BYTES = BQ * DQK * 2;
  static constexpr int DO_BYTES = FWD ? 0 : BQ * DV * 2;
  static constexpr int K_BYTES = BK * DQK * 2;
  static constexpr int V_BYTES = BK * DV * 2;
  // FWD row sum sum_j P: from the tensor core, a 64-column block of ones after V in every stage
  // (P.[V | 1]), or -- head dim 128, whose O and 16 more columns would not leave two CTAs room in
  // TMEM -- added up in fp32 by the softmax warpgroups
  static constexpr bool SUM_MMA = FWD && DQK != 128;
  static constexpr int ONES_BYTES = SUM_MMA ? BK * 128 : 0;
  static constexpr int STAGE_BYTES = K_BYTES + V_BYTES + ONES_BYTES;
  // CTAs per SM: the forward of head dims 64 and 128 fits two (half the shared memory and of
  // TMEM each), whose warps hide each other's latencies; every other variant runs one
  static constexpr int CTAS = (FWD && DQK <= 128) ? 2 : 1;
  static constexpr int BUDGET = CTAS == 2 ? 110 * 1024 : 220 * 1024;
  // Key/value staging: one ring of K + V (+ ones) stages; or, in the forward of head dims 128 (only
  // two such stages would fit) and 192 (three), separate rings: two V (+ ones) stages and as many
  // K stages as fit, so the first pass (K alone) and the P.V of the second do not hold the keys the
  // next S needs
  static constexpr int KST_RAW = (BUDGET - Q_BYTES - DO_BYTES) / STAGE_BYTES;
  static constexpr bool SPLIT = FWD && (KST_RAW < 3 || DQK == 192);
  static constexpr int VSTAGE_BYTES = V_BYTES + ONES_BYTES;  // one stage of the V ring
  static constexpr int VST = SPLIT ? 2 : 0;                  // V ring (SPLIT)
  static constexpr int KST_SPLIT = (BUDGET - Q_BYTES - DO_BYTES - VST * VSTAGE_BYTES) / K_BYTES;
  static constexpr int KST = SPLIT ? (KST_SPLIT > 8 ? 8 : KST_SPLIT)    // K ring (SPLIT)
                                   : (KST_RAW > 8 ? 8 : KST_RAW);       // or K + V ring
  static constexpr int SMEM =
      1024 + Q_BYTES + DO_BYTES + (SPLIT ? KST * K_BYTES + VST * VSTAGE_BYTES : KST * STAGE_BYTES);
  // TMEM: buffer b at b*BUF holds S (BK columns; P / dS packed over its first half) and, for
  // DQ, dP right after it; the accumulator (O or dQ) follows the NBUF buffers
  // (the MMA warp issues S of tile it + NBUF before the accumulation of tile it + 1: the key stages
  // must hold NBUF tiles and then some, or that S waits for a stage that the accumulation of tile
  // it has only just freed, and the accumulation of tile it + 1 waits behind it; keys in a ring of
  // their own are freed by S alone, so there NBUF stages suffice)
  static constexpr int NBUF = (FWD && KST >= (SPLIT ? 4 : 6)) ? 4 : 2;
  static constexpr uint32_t BUF = FWD ? BK : 2 * BK;
  static constexpr uint32_t T_ACC = NBUF * BUF;
  static constexpr uint32_t ACC_COLS = FWD ? DV + (SUM_MMA ? 16 : 0) : DQK;  // O [and 16 columns of row sum]
  static constexpr uint32_t OUT_COLS = FWD ? DV : DQK;       // columns written out
  static constexpr uint32_t TMEM_COLS = (T_ACC + ACC_COLS <= 256) ? 256 : 512;
  static constexpr int THREADS = 320;
  static_assert(KST >= 2 && NBUF <= KST, "stages");
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(T_ACC + ACC_COLS <= 512, "tmem");
  static_assert(CTAS == 1 || (TMEM_COLS <= 256 && SMEM <= 112 * 1024), "two CTAs per SM");
  static_assert(OUT_COLS % 64 == 0, "each warpgroup drains whole 32-column chunks");
};

struct QSmemCtl {
  uint64_t bar_q;
  uint64_t kv_full[8], kv_empty[8];  // K + V stages (K stages of the split rings)
  uint64_t v_full[2], v_empty[2];    // V stages of the split rings
  uint64_t s_full[4];   // tensor core -> warpgroup: S (and dP) of the buffer's tile are in TMEM
  uint64_t sm_done[4];  // warpgroup -> tensor core: S read / P or dS stored, buffer reusable
  uint64_t acc_done;
  uint32_t tmem_base;
  int abort_flag;
  float stat_m[2][128];  // FWD: each warpgroup's row maxima, combined once
  float stat_l[2][128];  // FWD without SUM_MMA: each warpgroup's row sums
};


template <int DQK, int DV, bool BF16, bool FWD>
__global__ void __launch_bounds__(320, (QCfg<DQK, DV, FWD>::CTAS))
    q_kernel(const Problem p, const __grid_constant__ Maps m, const float* __restrict__ sink, void* __restrict__ out,
             float* __restrict__ lse_out) {
  using C = QCfg<DQK, DV, FWD>;
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  extern __shared__ uint8_t smem_raw[];
  __shared__ QSmemCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sDO = sQ + C::Q_BYTES;
  uint8_t* sK0 = sDO + C::DO_BYTES;  // stage st: K at sK0 + st*STAGE_BYTES, V right after K
  uint8_t* sV0 = sK0 + C::KST * C::K_BYTES;  // SPLIT: K stage st at sK0 + st*K_BYTES, V stages from sV0
  constexpr int K_STRIDE = C::SPLIT ? C::K_BYTES : C::STAGE_BYTES;

  const int h = blockIdx.x;
  const int s = blockIdx.z;
  Seq sq, sk;  // the sequence's queries and keys
  if (!load_seq(p, s, sq) || !load_kseq(p, s, sk)) return;
  const int off = sk.len - sq.len;  // query i sits on key diagonal i + off
  const int ntq = (sq.len + C::BQ - 1) / C::BQ;
  const int t = static_cast<int>(gridDim.y) - 1 - static_cast<int>(blockIdx.y);  // heavy tiles first
  if (t >= ntq) return;
  int k0, k1;
  kv_tiles_for_q_tile(t, sq.len, sk.len, C::BK, p.right, p.window, &k0, &k1);
  const int n = k1 - k0;
  const int NIT = FWD ? 2 * n : n;
  const int g = h / p.G;
  const int zq = sq.b * p.Hq + h;  // row block of the contiguous fp32 [B, Hq, S] LSE
  const int row0 = sq.start + t * C::BQ;

  // the warp index goes through a shuffle so the compiler knows it is warp-uniform: the warp-role
  // branches below are then uniform and the MMA operands can stay in uniform registers
  const int tid = threadIdx.x, warp = __shfl_sync(0xffffffffu, tid >> 5, 0), lane = tid & 31;
  if (tid == 0) {
    mbar_init(&ctl.bar_q, 1);
    for (int i = 0; i < C::KST; ++i) {
      mbar_init(&ctl.kv_full[i], 1);
      mbar_init(&ctl.kv_empty[i], 1);
    }
    for (int i = 0; i < C::VST; ++i) {
      mbar_init(&ctl.v_full[i], 1);
      mbar_init(&ctl.v_empty[i], 1);
    }
    for (int i = 0; i < C::NBUF; ++i) {
      mbar_init(&ctl.s_full[i], 1);
      mbar_init(&ctl.sm_done[i], 4);  // one arrival per warp of the warpgroup
    }
    mbar_init(&ctl.acc_done, 1);
    ctl.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(&ctl.tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (C::SUM_MMA) {
    // the constant ones blocks (TMA never writes them); 1.0 in the input dtype
    const uint32_t one2 = BF16 ? 0x3F803F80u : 0x3C003C00u;
    for (int st = 0; st < (C::SPLIT ? C::VST : C::KST); ++st) {
      uint8_t* v = C::SPLIT ? sV0 + st * C::VSTAGE_BYTES : sK0 + st * C::STAGE_BYTES + C::K_BYTES;
      uint4* blk = reinterpret_cast<uint4*>(v + C::V_BYTES);
      for (int i = tid; i < C::ONES_BYTES / 16; i += C::THREADS) blk[i] = make_uint4(one2, one2, one2, one2);
    }
    fence_async_smem();  // generic-proxy writes read later by the tensor core
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // broadcast from lane 0 so the compiler treats the TMEM base as warp-uniform
  const uint32_t tmem = __shfl_sync(0xffffffffu, ctl.tmem_base, 0);
  const WaitGuard guard{p.err, &ctl.abort_flag, p.wait_limit};

  if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_map(&m.q);
      tma_prefetch_map(&m.k);
      tma_prefetch_map(&m.v);
      mbar_expect_tx(&ctl.bar_q, C::Q_BYTES + C::DO_BYTES);
      for (int cb = 0; cb < C::QB; ++cb) tma_load_4d(sQ + cb * (C::BQ * 128), &m.q, &ctl.bar_q, cb * 64, row0, h, sq.b);
      if (!FWD)
        for (int cb = 0; cb < C::VB; ++cb)
          tma_load_4d(sDO + cb * (C::BQ * 128), &m.dout, &ctl.bar_q, cb * 64, row0, h, sq.b);
      int issued = 0, issued_v = 0;
      if constexpr (C::SPLIT) {
        // K of tile i, then V of tile i - (NBUF - 1) (when it is a second-pass tile): the order in
        // which the MMA warp consumes them (S of tile i + NBUF follows P.V of tile i)
        for (int i = 0; i <= NIT + C::NBUF - 2; ++i) {
          if (i < NIT) {
            const int st = i % C::KST;
            if (i >= C::KST && !mbar_wait(&ctl.kv_empty[st], ((i / C::KST) - 1) & 1, guard, 1)) break;
            uint8_t* sK = sK0 + st * C::K_BYTES;
            const int krow = sk.start + (k0 + i % n) * C::BK;
            mbar_expect_tx(&ctl.kv_full[st], C::K_BYTES);
            for (int cb = 0; cb < C::QB; ++cb)
              tma_load_4d(sK + cb * (C::BK * 128), &m.k, &ctl.kv_full[st], cb * 64, krow, g, sk.b);
            issued = i + 1;
          }
          const int vi = i - (C::NBUF - 1) - n;  // second-pass index of that tile (key tile k0 + vi)
          if (vi >= 0 && vi < n) {
            const int vs = vi % C::VST;
            if (vi >= C::VST && !mbar_wait(&ctl.v_empty[vs], ((vi / C::VST) - 1) & 1, guard, 1)) break;
            uint8_t* sV = sV0 + vs * C::VSTAGE_BYTES;
            const int krow = sk.start + (k0 + vi) * C::BK;
            mbar_expect_tx(&ctl.v_full[vs], C::V_BYTES);
            for (int cb = 0; cb < C::VB; ++cb)
              tma_load_4d(sV + cb * (C::BK * 128), &m.v, &ctl.v_full[vs], cb * 64, krow, g, sk.b);
            issued_v = vi + 1;
          }
        }
      } else for (int it = 0; it < NIT; ++it) {
        const int st = it % C::KST;
        if (it >= C::KST && !mbar_wait(&ctl.kv_empty[st], ((it / C::KST) - 1) & 1, guard, 1)) break;
        const bool need_v = !FWD || it >= n;
        const int kt = k0 + (FWD ? it % n : it);
        uint8_t* sK = sK0 + st * C::STAGE_BYTES;
        uint8_t* sV = sK + C::K_BYTES;
        mbar_expect_tx(&ctl.kv_full[st], C::K_BYTES + (need_v ? C::V_BYTES : 0));
        const int krow = sk.start + kt * C::BK;
        for (int cb = 0; cb < C::QB; ++cb)
          tma_load_4d(sK + cb * (C::BK * 128), &m.k, &ctl.kv_full[st], cb * 64, krow, g, sk.b);
        if (need_v)
          for (int cb = 0; cb < C::VB; ++cb)
            tma_load_4d(sV + cb * (C::BK * 128), &m.v, &ctl.kv_full[st], cb * 64, krow, g, sk.b);
        issued = it + 1;
      }
      if (ctl.abort_flag) {
        // let copies already in flight land before the CTA's shared memory goes away
        volatile int no_abort = 0;
        const WaitGuard g2{nullptr, &no_abort, p.wait_limit};
        mbar_wait(&ctl.bar_q, 0, g2, 0);
        for (int it = issued - C::KST < 0 ? 0 : issued - C::KST; it < issued; ++it)
          mbar_wait(&ctl.kv_full[it % C::KST], (it / C::KST) & 1, g2, 0);
        if constexpr (C::SPLIT)
          for (int vi = issued_v - C::VST < 0 ? 0 : issued_v - C::VST; vi < issued_v; ++vi)
            mbar_wait(&ctl.v_full[vi % C::VST], (vi / C::VST) & 1, g2, 0);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    {  // the whole warp runs the issue loop; one elected lane issues each MMA
      constexpr uint32_t idS = idesc_f16(128, C::BK, BF16, false, false);
      constexpr uint32_t idPV = idesc_f16(128, DV + (C::SUM_MMA ? 16 : 0), BF16, false, true);  // P.[V | 1]
      constexpr uint32_t idDQ = idesc_f16(128, DQK, BF16, false, true);
      const uint64_t dQ0 = sdesc_sw128(smem_u32(sQ), 16, 1024);    // Q, K-major (A of S)
      const uint64_t dDO0 = sdesc_sw128(smem_u32(sDO), 16, 1024);  // dO, K-major (A of dP)
      auto kstep = [](int kk, int rows) -> uint32_t { return (kk / 4) * (rows * 128) + (kk % 4) * 32; };
      bool ok = mbar_wait_warp(&ctl.bar_q, 0, guard, 2);
      // S (and dP) of tile `it` into buffer it % NBUF, once the tile NBUF earlier has left it
      auto issue_s = [&](int it) -> bool {
        const int st = it % C::KST, b = it % C::NBUF;
        if (!mbar_wait_warp(&ctl.kv_full[st], (it / C::KST) & 1, guard, 3)) return false;
        if (it >= C::NBUF && !mbar_wait_warp(&ctl.sm_done[b], ((it - C::NBUF) / C::NBUF) & 1, guard, 4))
          return false;
        tc_fence_after();
        const uint32_t aK = smem_u32(sK0 + st * K_STRIDE);
        const uint64_t dK = sdesc_sw128(aK, 16, 1024);
        const uint32_t tS = tmem + b * C::BUF;
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk)
          umma_ss(tS, desc_advance(dQ0, kstep(kk, C::BQ)), desc_advance(dK, kstep(kk, C::BK)), idS, kk > 0);
        if (!FWD) {
          const uint64_t dV = sdesc_sw128(aK + C::K_BYTES, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < DV / 16; ++kk)
            umma_ss(tS + C::BK, desc_advance(dDO0, kstep(kk, C::BQ)), desc_advance(dV, kstep(kk, C::BK)), idS,
                    kk > 0);
        }
        umma_commit(&ctl.s_full[b]);
        // statistics pass, or keys of their own ring: K consumed by S alone
        if (C::SPLIT || (FWD && it < n)) umma_commit(&ctl.kv_empty[st]);
        return true;
      };
      // FWD: O += P.V; DQ: dQ += dS.K -- A = the packed P / dS in the tile's buffer
      auto issue_acc = [&](int it) -> bool {
        const int st = it % C::KST, b = it % C::NBUF;
        constexpr int VSTN = C::VST > 0 ? C::VST : 1;
        const int vi = it - n, vs = C::SPLIT ? vi % VSTN : 0;  // SPLIT: V of second-pass tile vi
        if (!mbar_wait_warp(&ctl.sm_done[b], (it / C::NBUF) & 1, guard, 5)) return false;
        if (C::SPLIT && !mbar_wait_warp(&ctl.v_full[vs], (vi / VSTN) & 1, guard, 8)) return false;
        tc_fence_after();
        const uint32_t aK = smem_u32(sK0 + st * K_STRIDE);
        const uint32_t tA = tmem + b * C::BUF;
        const int first = FWD ? n : 0;
        if (FWD) {
          // [V | ones], MN-major (B of P.[V | 1]): the ones block follows V's 64-column blocks
          const uint32_t aV = C::SPLIT ? smem_u32(sV0 + vs * C::VSTAGE_BYTES) : aK + C::K_BYTES;
          const uint64_t dVmn = sdesc_sw128(aV, C::BK * 128, 1024);
#pragma unroll
          for (int kk = 0; kk < C::BK / 16; ++kk)
            umma_ts(tmem + C::T_ACC, tA + kk * 8, desc_advance(dVmn, kk * 2048), idPV,
                    (it > first || kk > 0) ? 1u : 0u);
        } else {
          const uint64_t dKmn = sdesc_sw128(aK, C::BK * 128, 1024);  // K, MN-major (B of dS.K)
#pragma unroll
          for (int kk = 0; kk < C::BK / 16; ++kk)
            umma_ts(tmem + C::T_ACC, tA + kk * 8, desc_advance(dKmn, kk * 2048), idDQ,
                    (it > first || kk > 0) ? 1u : 0u);
        }
        umma_commit(C::SPLIT ? &ctl.v_empty[vs] : &ctl.kv_empty[st]);
        return true;
      };
      for (int it = 0; ok && it < C::NBUF && it < NIT; ++it) ok = issue_s(it);
      // in the order the warpgroups release the buffers: tile it's accumulation, then the
      // tile that takes its buffer next
      for (int it = 0; ok && it < NIT; ++it) {
        if ((!FWD || it >= n) && !issue_acc(it)) break;
        if (it + C::NBUF < NIT && !issue_s(it + C::NBUF)) break;
      }
      umma_commit(&ctl.acc_done);
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int w = warp >> 2;  // which tiles: index parity w
    const int r = tid & 127;  // query row within the tile == TMEM lane
    const int il = t * C::BQ + r;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float sl2 = p.scale_log2;
    const float2 sl22 = make_float2(sl2, sl2);
    bool ok = true;
    if (FWD) {
      float mx = -INFINITY;  // running maximum of this warpgroup's logits (log2 units)
      const float sink2 = sink ? __ldg(sink + h) * kLog2e : -INFINITY;
      if (w == 0) mx = sink2;
      float mref = 0.f;  // the row maximum both passes agree on (0 for a row with no allowed key)
      float lsum = 0.f;  // without SUM_MMA: this warpgroup's share of sum_j P
      bool combined = false;
      // both warpgroups' maxima -> the row maximum (once, before the first output tile)
      auto combine = [&]() {
        ctl.stat_m[w][r] = mx;
        named_bar_sync(1, 256);
        const float M = fmaxf(ctl.stat_m[0][r], ctl.stat_m[1][r]);
        mref = (M == -INFINITY) ? 0.f : M;
        combined = true;
      };
      for (int it = w; it < NIT; it += 2) {
        const int kt = k0 + it % n;
        const int j0 = kt * C::BK;
        const bool need_mask = (j0 + C::BK > sk.len) || (p.right > 0 && j0 + C::BK > t * C::BQ + off + p.right) ||
                               (p.window > 0 && t * C::BQ + C::BQ - 1 + off - j0 >= p.window);
        if (it >= n && !combined) combine();
        const int b = it % C::NBUF;
        const uint32_t tS = tmem + lane_base + b * C::BUF;
        if (!mbar_wait_warp(&ctl.s_full[b], (it / C::NBUF) & 1, guard, 6)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t v[C::BK];
        tmem_ld64(tS, v);
        if (it < n) {
          // first pass: the row maximum of the raw logits (scale > 0 commutes with max)
          float c0 = -INFINITY, c1 = -INFINITY;
#pragma unroll
          for (int e = 0; e < C::BK; e += 2) {
            float a = __uint_as_float(v[e]), b = __uint_as_float(v[e + 1]);
            if (need_mask) {
              const int d0 = il + off - j0;  // diagonal distance to this tile's first key
              if (!visible_d(d0 - e, j0 + e < sk.len, p.right, p.window)) a = -INFINITY;
              if (!visible_d(d0 - e - 1, j0 + e + 1 < sk.len, p.right, p.window)) b = -INFINITY;
            }
            c0 = fmaxf(c0, a);
            c1 = fmaxf(c1, b);
          }
          mx = fmaxf(mx, fmaxf(c0, c1) * sl2);
          tc_fence_before();
        } else {
          // second pass: P = exp2(S*scale*log2e - max) <= 1, packed in place over S
          uint32_t pk[C::BK / 2];
          const float2 nl = make_float2(-mref, -mref);
          if constexpr (!C::SUM_MMA) {
            // P in fp32, masked, added up (four partial sums) and packed
            float s4[4] = {0.f, 0.f, 0.f, 0.f};
            const int d0 = il + off - j0;  // diagonal distance to this tile's first key
#pragma unroll
            for (int e = 0; e < C::BK; e += 2) {
              const float2 x = fma2(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), sl22, nl);
              float pa = ex2_approx(x.x), pb = ex2_approx(x.y);
              if (need_mask) {
                if (!visible_d(d0 - e, j0 + e < sk.len, p.right, p.window)) pa = 0.f;
                if (!visible_d(d0 - e - 1, j0 + e + 1 < sk.len, p.right, p.window)) pb = 0.f;
              }
              s4[(e >> 1) & 3] += pa + pb;
              pk[e / 2] = pack2<BF16>(pa, pb);
            }
            lsum += (s4[0] + s4[1]) + (s4[2] + s4[3]);
          } else {
#pragma unroll
          for (int e = 0; e < C::BK; e += 4) {
            const float2 x0 = fma2(make_float2(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), sl22, nl);
            const float2 x1 = fma2(make_float2(__uint_as_float(v[e + 2]), __uint_as_float(v[e + 3])), sl22, nl);
            if (BF16) {
              pk[e / 2] = pack2<true>(ex2_approx(x0.x), ex2_approx(x0.y));
              pk[e / 2 + 1] = pack2<true>(ex2_approx(x1.x), ex2_approx(x1.y));
            } else {
              // the argument rounded to fp16, exponentiated two at a time (adds at most ~2e-4 to P)
              pk[e / 2] = ex2_f16x2(pack2<false>(x0.x, x0.y));
              pk[e / 2 + 1] = ex2_f16x2(pack2<false>(x1.x, x1.y));
            }
          }
          if (need_mask) {
#pragma unroll
            for (int e = 0; e < C::BK; ++e)
              if (!visible_d(il + off - j0 - e, j0 + e < sk.len, p.right, p.window))
                pk[e / 2] &= (e & 1) ? 0x0000FFFFu : 0xFFFF0000u;
          }
          }
          uint32_t p0[16], p1[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            p0[e] = pk[e];
            p1[e] = pk[16 + e];
          }
          tmem_st16(tS, p0);
          tmem_st16(tS + 16, p1);
          tmem_st_wait();
          tc_fence_before();
        }
        mbar_arrive_warp(&ctl.sm_done[b]);
      }
      if (!combined) combine();  // both warpgroups reach the named barrier exactly once
      float lrow = 0.f;
      if constexpr (!C::SUM_MMA) {  // the two warpgroups' row sums (again once each, unconditionally)
        ctl.stat_l[w][r] = lsum;
        named_bar_sync(1, 256);
        lrow = ctl.stat_l[0][r] + ctl.stat_l[1][r];
      }
      // epilogue: l = sum_j P (the ones column, or the warpgroups' sums) + the sink's term;
      // O = (P.V) / l; LSE = max + log l.  Warpgroup w writes output columns [w*DV/2, (w+1)*DV/2)
      if (ok && mbar_wait_warp(&ctl.acc_done, 0, guard, 7)) {
        tc_fence_after();
        const bool valid = il < sq.len;
        const size_t orow = (static_cast<size_t>(zq) * p.S + sq.start + il);
        float l = lrow;
        if (C::SUM_MMA && n > 0) {
          uint32_t sv[16];
          tmem_ld16(tmem + lane_base + C::T_ACC + DV, sv);
          l = __uint_as_float(sv[0]);
        }
        if (sink2 != -INFINITY) l += ex2_approx(sink2 - mref);
        const float inv = l > 0.f ? 1.f / l : 0.f;
        T* o = static_cast<T*>(out) + p.o_st.row(sq.b, h, sq.start + il);
#pragma unroll 1
        for (int c0 = w * (DV / 2); c0 < (w + 1) * (DV / 2); c0 += 32) {
          uint32_t v[32];
          if (n > 0) tmem_ld32(tmem + lane_base + C::T_ACC + c0, v);
          else
            for (int e = 0; e < 32; ++e) v[e] = 0u;
          if (valid) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint4 u;
              u.x = pack2<BF16>(__uint_as_float(v[8 * q4 + 0]) * inv, __uint_as_float(v[8 * q4 + 1]) * inv);
              u.y = pack2<BF16>(__uint_as_float(v[8 * q4 + 2]) * inv, __uint_as_float(v[8 * q4 + 3]) * inv);
              u.z = pack2<BF16>(__uint_as_float(v[8 * q4 + 4]) * inv, __uint_as_float(v[8 * q4 + 5]) * inv);
              u.w = pack2<BF16>(__uint_as_float(v[8 * q4 + 6]) * inv, __uint_as_float(v[8 * q4 + 7]) * inv);
              *reinterpret_cast<uint4*>(o + c0 + 8 * q4) = u;
            }
          }
        }
        if (valid && w == 0) lse_out[orow] = (l > 0.f) ? (mref + log2f(l)) * kLn2 : -INFINITY;
      }
    } else {
      // query-stationary dQ pass
      const size_t sidx = stat_index(p, h, s, t) + r;
      const float nlse2 = p.nlse2[sidx];
      const float ndlt = p.ndelta[sidx];
      for (int it = w; it < NIT; it += 2) {
        const int kt = k0 + it;
        const int j0 = kt * C::BK;
        const bool need_mask = (j0 + C::BK > sk.len) || (p.right > 0 && j0 + C::BK > t * C::BQ + off + p.right) ||
                               (p.window > 0 && t * C::BQ + C::BQ - 1 + off - j0 >= p.window);
        const int b = it % C::NBUF;
        const uint32_t tS = tmem + lane_base + b * C::BUF;
        if (!mbar_wait_warp(&ctl.s_full[b], (it / C::NBUF) & 1, guard, 6)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < C::BK; c0 += 32) {
          uint32_t sv[32], dv[32];
          tmem_ld32(tS + c0, sv);
          tmem_ld32(tS + C::BK + c0, dv);
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float pa = ex2_approx(fmaf(__uint_as_float(sv[2 * e]), sl2, nlse2));
            float pb = ex2_approx(fmaf(__uint_as_float(sv[2 * e + 1]), sl2, nlse2));
            if (need_mask) {
              const int d0 = il + off - j0 - c0;  // diagonal distance to this chunk's first key
              if (!visible_d(d0 - 2 * e, j0 + c0 + 2 * e < sk.len, p.right, p.window)) pa = 0.f;
              if (!visible_d(d0 - 2 * e - 1, j0 + c0 + 2 * e + 1 < sk.len, p.right, p.window)) pb = 0.f;
            }
            const float da = pa * (__uint_as_float(dv[2 * e]) + ndlt);
            const float db = pb * (__uint_as_float(dv[2 * e + 1]) + ndlt);
            pk[e] = pack2<BF16>(da, db);
          }
          // dS packed over S's first half: chunk c0 lands in columns [c0/2, c0/2 + 16), already read
          tmem_st16(tS + c0 / 2, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(&ctl.sm_done[b]);
      }
      // epilogue: dQ (x scale); warpgroup w writes columns [w*DQK/2, (w+1)*DQK/2)
      if (ok && mbar_wait_warp(&ctl.acc_done, 0, guard, 7)) {
        tc_fence_after();
        const bool valid = il < sq.len;
        T* dq = static_cast<T*>(out) + p.dq_st.row(sq.b, h, sq.start + il);
#pragma unroll 1
        for (int c0 = w * (DQK / 2); c0 < (w + 1) * (DQK / 2); c0 += 32) {
          uint32_t v[32];
          if (n > 0) tmem_ld32(tmem + lane_base + C::T_ACC + c0, v);  // all lanes: .sync.aligned
          else
            for (int e = 0; e < 32; ++e) v[e] = 0u;
          if (!valid) continue;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 u;
            u.x = pack2<BF16>(__uint_as_float(v[8 * q4 + 0]) * p.scale, __uint_as_float(v[8 * q4 + 1]) * p.scale);
            u.y = pack2<BF16>(__uint_as_float(v[8 * q4 + 2]) * p.scale, __uint_as_float(v[8 * q4 + 3]) * p.scale);
            u.z = pack2<BF16>(__uint_as_float(v[8 * q4 + 4]) * p.scale, __uint_as_float(v[8 * q4 + 5]) * p.scale);
            u.w = pack2<BF16>(__uint_as_float(v[8 * q4 + 6]) * p.scale, __uint_as_float(v[8 * q4 + 7]) * p.scale);
            *reinterpret_cast<uint4*>(dq + c0 + 8 * q4) = u;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int DQK, int DV, bool BF16, bool FWD>
static cudaError_t launch_q_t(const Problem& p, const Maps& m, const float* sink, void* out, float* lse,
                              cudaStream_t st) {
  using C = QCfg<DQK, DV, FWD>;
  auto kern = q_kernel<DQK, DV, BF16, FWD>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int ntiles = (p.max_len + C::BQ - 1) / C::BQ;
  if (ntiles == 0 || p.nseqs == 0) return cudaSuccess;
  dim3 grid(p.Hq, ntiles, p.nseqs);
  kern<<<grid, C::THREADS, C::SMEM, st>>>(p, m, sink, out, lse);
  return cudaGetLastError();
}

template <bool FWD>
static cudaError_t dispatch_q(const Problem& p, int bf16, const Maps& m, const float* sink, void* out, float* lse,
                              cudaStream_t st) {
#define GQA_Q(DQK, DV)                                                              \
  if (p.Dqk == DQK && p.Dv == DV)                                                   \
    return bf16 ? launch_q_t<DQK, DV, true, FWD>(p, m, sink, out, lse, st)           \
                : launch_q_t<DQK, DV, false, FWD>(p, m, sink, out, lse, st);
  GQA_Q(64, 64)
  GQA_Q(128, 128)
  GQA_Q(192, 128)
#undef GQA_Q
  return cudaErrorInvalidValue;
}

cudaError_t launch_dq(const Problem& p, int dtype_bf16, const Maps& m, void* dq, cudaStream_t st) {
  return dispatch_q<false>(p, dtype_bf16, m, nullptr, dq, nullptr, st);
}

int q_kernel_bk() { return QCfg<64, 64, true>::BK; }

}  // namespace gqa
