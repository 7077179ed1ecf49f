// Query-stationary tcgen05 kernels: one CTA owns 128 query rows of one query
// head and streams the 128-row key/value tiles it can see.
//
//   FWD : forward with causal / sliding-window / attention-sink masking
//         (tilelang-ascend PR #1638 "Add GQA Sink Backward BHSD", 4->2 commit:
//         "flashattn_fwd: online softmax + sink + window -> O, lse").  Two passes
//         over the key tiles: the first forms the row statistics (running max and
//         sum, sink included), the second forms P = exp(S - LSE) already
//         normalised and accumulates O = P.V in TMEM, so O is never rescaled.
//   DQ  : the deterministic dQ pass: S = Q.K^T, dP = dO.V^T, dS = P*(dP - Delta)
//         (same PR, review thread k1..k5, in the query-stationary loop order the
//         Ascend kernel uses for dQ, "dQ[L0C accumulate]"); dQ = scale * dS.K
//         accumulates in TMEM with no atomics.
//
// Warp roles (192 threads): warps 0-3 = softmax warpgroup, thread r owns query
// row r = TMEM lane r; warp 4 = TMA producer; warp 5 = TMEM allocator + MMA
// issuer (one elected thread).  Operands live in shared memory in the 128-byte
// swizzled layout TMA writes; S, dP, O, dQ accumulate in TMEM; P / dS are packed
// to 16-bit in TMEM and feed the next MMA as its A operand.
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <type_traits>
#include "common.cuh"
#include "umma.cuh"
#include "launch.h"

namespace gqa {

template <int DQK, int DV, bool FWD>
struct QCfg {
  static constexpr int BQ = 128, BK = 128;
  static constexpr int QB = DQK / 64, VB = DV / 64;  // 64-column (128-byte) blocks
  static constexpr int Q_BYTES = BQ * DQK * 2;
  static constexpr int DO_BYTES = FWD ? 0 : BQ * DV * 2;
  static constexpr int K_BYTES = BK * DQK * 2;
  static constexpr int V_BYTES = BK * DV * 2;
  static constexpr int STAGE_BYTES = K_BYTES + V_BYTES;
  static constexpr int BUDGET = 220 * 1024;
  static constexpr int KST_RAW = (BUDGET - Q_BYTES - DO_BYTES) / STAGE_BYTES;
  static constexpr int KST = KST_RAW > 4 ? 4 : (KST_RAW < 1 ? 1 : KST_RAW);
  static constexpr int SMEM = 1024 + Q_BYTES + DO_BYTES + KST * STAGE_BYTES;
  // TMEM columns
  static constexpr uint32_t T_S0 = 0, T_S1 = 128;         // FWD: two S buffers; DQ: S and dP
  static constexpr uint32_t T_ACC = 256;                  // FWD: O; DQ: dQ
  static constexpr int THREADS = 192;
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(T_ACC + (FWD ? DV : DQK) <= 512, "tmem");
};

struct QSmemCtl {
  uint64_t bar_q;
  uint64_t kv_full[4], kv_empty[4];
  uint64_t s_full[2], s_free[2], p_full[2];
  uint64_t acc_done;
  uint32_t tmem_base;
  int abort_flag;
};

// Allowed-key test for query row i (local) and key j (local).
__device__ __forceinline__ bool allowed(int i, int j, int len, int causal, int window) {
  return j < len && (!causal || j <= i) && (window <= 0 || i - j < window);
}

template <int DQK, int DV, bool BF16, bool FWD>
__global__ void __launch_bounds__(192, 1)
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

  const int h = blockIdx.x;
  const int s = blockIdx.z;
  Seq sq;
  if (!load_seq(p, s, sq)) return;
  const int ntq = (sq.len + C::BQ - 1) / C::BQ;
  const int t = static_cast<int>(gridDim.y) - 1 - static_cast<int>(blockIdx.y);  // heavy tiles first
  if (t >= ntq) return;
  int k0, k1;
  kv_tiles_for_q_tile(t, sq.len, p.causal, p.window, &k0, &k1);
  const int n = k1 - k0;
  const int NIT = FWD ? 2 * n : n;
  const int g = h / p.G;
  const int zq = sq.b * p.Hq + h, zk = sq.b * p.Hkv + g;
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
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl.s_full[i], 1);
      mbar_init(&ctl.s_free[i], 4);  // one arrival per softmax warp
      mbar_init(&ctl.p_full[i], 4);
    }
    mbar_init(&ctl.acc_done, 1);
    ctl.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&ctl.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // broadcast from lane 0 so the compiler treats the TMEM base as warp-uniform (uniform registers
  // for the MMA operands instead of per-MMA register moves)
  const uint32_t tmem = __shfl_sync(0xffffffffu, ctl.tmem_base, 0);
  const WaitGuard guard{p.err, &ctl.abort_flag, p.wait_limit};

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_map(&m.q);
      tma_prefetch_map(&m.k);
      tma_prefetch_map(&m.v);
      mbar_expect_tx(&ctl.bar_q, C::Q_BYTES + C::DO_BYTES);
      for (int cb = 0; cb < C::QB; ++cb) tma_load_3d(sQ + cb * (C::BQ * 128), &m.q, &ctl.bar_q, cb * 64, row0, zq);
      if (!FWD)
        for (int cb = 0; cb < C::VB; ++cb)
          tma_load_3d(sDO + cb * (C::BQ * 128), &m.dout, &ctl.bar_q, cb * 64, row0, zq);
      int issued = 0;
      for (int it = 0; it < NIT; ++it) {
        const int st = it % C::KST;
        if (it >= C::KST && !mbar_wait(&ctl.kv_empty[st], ((it / C::KST) - 1) & 1, guard, 1)) break;
        const bool need_v = !FWD || it >= n;
        const int kt = k0 + (FWD ? it % n : it);
        uint8_t* sK = sK0 + st * C::STAGE_BYTES;
        uint8_t* sV = sK + C::K_BYTES;
        mbar_expect_tx(&ctl.kv_full[st], C::K_BYTES + (need_v ? C::V_BYTES : 0));
        const int krow = sq.start + kt * C::BK;
        for (int cb = 0; cb < C::QB; ++cb)
          tma_load_3d(sK + cb * (C::BK * 128), &m.k, &ctl.kv_full[st], cb * 64, krow, zk);
        if (need_v)
          for (int cb = 0; cb < C::VB; ++cb)
            tma_load_3d(sV + cb * (C::BK * 128), &m.v, &ctl.kv_full[st], cb * 64, krow, zk);
        issued = it + 1;
      }
      if (ctl.abort_flag) {
        // let copies already in flight land before the CTA's shared memory goes away
        volatile int no_abort = 0;
        const WaitGuard g2{nullptr, &no_abort, p.wait_limit};
        mbar_wait(&ctl.bar_q, 0, g2, 0);
        for (int it = issued - C::KST < 0 ? 0 : issued - C::KST; it < issued; ++it)
          mbar_wait(&ctl.kv_full[it % C::KST], (it / C::KST) & 1, g2, 0);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    {  // the whole warp runs the issue loop; one elected lane issues each MMA
      constexpr uint32_t idS = idesc_f16(128, C::BK, BF16, false, false);
      constexpr uint32_t idPV = idesc_f16(128, DV, BF16, false, true);
      constexpr uint32_t idDQ = idesc_f16(128, DQK, BF16, false, true);
      const uint32_t aQ = smem_u32(sQ), aDO = smem_u32(sDO);
      bool ok = mbar_wait_warp(&ctl.bar_q, 0, guard, 2);
      int pending = -1;  // output-pass tile whose P.V is not issued yet
      auto issue_pv = [&](int j) -> bool {
        const int u = j - n;
        if (!mbar_wait_warp(&ctl.p_full[u & 1], (u >> 1) & 1, guard, 5)) return false;
        tc_fence_after();
        const uint32_t tP = tmem + ((j & 1) ? C::T_S1 : C::T_S0);
        const uint32_t aVj = smem_u32(sK0 + (j % C::KST) * C::STAGE_BYTES) + C::K_BYTES;
#pragma unroll
        for (int kk = 0; kk < C::BK / 16; ++kk)
          umma_ts(tmem + C::T_ACC, tP + kk * 8, sdesc_sw128(aVj + kk * 2048, C::BK * 128, 1024), idPV,
                  (u > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&ctl.kv_empty[j % C::KST]);
        return true;
      };
      for (int it = 0; ok && it < NIT; ++it) {
        const int st = it % C::KST;
        const uint32_t aK = smem_u32(sK0 + st * C::STAGE_BYTES);
        const uint32_t aV = aK + C::K_BYTES;
        if (!mbar_wait_warp(&ctl.kv_full[st], (it / C::KST) & 1, guard, 3)) break;
        if (FWD) {
          const int buf = it & 1;
          if (it >= 2 && !mbar_wait_warp(&ctl.s_free[buf], ((it - 2) >> 1) & 1, guard, 4)) break;
          tc_fence_after();
          const uint32_t tS = tmem + (buf ? C::T_S1 : C::T_S0);
#pragma unroll
          for (int kk = 0; kk < DQK / 16; ++kk)
            umma_ss(tS, sdesc_sw128(aQ + (kk / 4) * (C::BQ * 128) + (kk % 4) * 32, 16, 1024),
                    sdesc_sw128(aK + (kk / 4) * (C::BK * 128) + (kk % 4) * 32, 16, 1024), idS, kk > 0);
          umma_commit(&ctl.s_full[buf]);
          if (it < n) umma_commit(&ctl.kv_empty[st]);  // statistics pass: K consumed by S alone
          // the P.V of the previous output-pass tile goes after this tile's S (one tile of lookahead)
          if (pending >= 0) {
            if (!issue_pv(pending)) break;
            pending = -1;
          }
          if (it >= n) pending = it;
        } else {
          if (it >= 1 && !mbar_wait_warp(&ctl.s_free[0], (it - 1) & 1, guard, 4)) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < DQK / 16; ++kk)
            umma_ss(tmem + C::T_S0, sdesc_sw128(aQ + (kk / 4) * (C::BQ * 128) + (kk % 4) * 32, 16, 1024),
                    sdesc_sw128(aK + (kk / 4) * (C::BK * 128) + (kk % 4) * 32, 16, 1024), idS, kk > 0);
#pragma unroll
          for (int kk = 0; kk < DV / 16; ++kk)
            umma_ss(tmem + C::T_S1, sdesc_sw128(aDO + (kk / 4) * (C::BQ * 128) + (kk % 4) * 32, 16, 1024),
                    sdesc_sw128(aV + (kk / 4) * (C::BK * 128) + (kk % 4) * 32, 16, 1024), idS, kk > 0);
          umma_commit(&ctl.s_full[0]);
          if (!mbar_wait_warp(&ctl.p_full[0], it & 1, guard, 5)) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < C::BK / 16; ++kk)
            umma_ts(tmem + C::T_ACC, tmem + C::T_S1 + kk * 8, sdesc_sw128(aK + kk * 2048, C::BK * 128, 1024),
                    idDQ, (it > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&ctl.kv_empty[st]);
        }
      }
      if (FWD && ok && pending >= 0) issue_pv(pending);
      umma_commit(&ctl.acc_done);
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroup
    const int r = tid;  // query row within the tile == TMEM lane
    const int il = t * C::BQ + r;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const float sl2 = p.scale_log2;
    bool ok = true;
    if (FWD) {
      float mx = -INFINITY, l = 0.f;  // running max (log2 units) and sum
      if (sink) {
        mx = __ldg(sink + h) * kLog2e;
        l = 1.f;
      }
      float lse2 = 0.f;
      for (int it = 0; it < NIT; ++it) {
        const int buf = it & 1;
        const int kt = k0 + it % n;
        const int j0 = kt * C::BK;
        const bool need_mask = (j0 + C::BK > sq.len) || (p.causal && j0 + C::BK - 1 > t * C::BQ) ||
                               (p.window > 0 && t * C::BQ + C::BQ - 1 - j0 >= p.window);
        if (!mbar_wait_warp(&ctl.s_full[buf], (it >> 1) & 1, guard, 6)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tS = tmem + lane_base + (buf ? C::T_S1 : C::T_S0);
        if (it < n) {
          // statistics pass
#pragma unroll 1
          for (int c0 = 0; c0 < C::BK; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tS + c0, v);
            float cm = -INFINITY;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              float x = __uint_as_float(v[e]) * sl2;
              if (need_mask && !allowed(il, j0 + c0 + e, sq.len, p.causal, p.window)) x = -INFINITY;
              v[e] = __float_as_uint(x);
              cm = fmaxf(cm, x);
            }
            const float mn = fmaxf(mx, cm);
            if (mn != -INFINITY) {
              float acc = 0.f;
#pragma unroll
              for (int e = 0; e < 32; ++e) acc += ex2_approx(__uint_as_float(v[e]) - mn);
              l = l * ex2_approx(mx - mn) + acc;
              mx = mn;
            }
          }
          tc_fence_before();
          mbar_arrive_warp(&ctl.s_free[buf]);
          if (it == n - 1) lse2 = (l > 0.f) ? mx + log2f(l) : INFINITY;
        } else {
          // output pass: P = exp2(S*scale*log2e - LSE2), packed in place over S
          const int u = it - n;
#pragma unroll 1
          for (int c0 = 0; c0 < C::BK; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tS + c0, v);
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float a = ex2_approx(fmaf(__uint_as_float(v[2 * e]), sl2, -lse2));
              float b = ex2_approx(fmaf(__uint_as_float(v[2 * e + 1]), sl2, -lse2));
              if (need_mask) {
                if (!allowed(il, j0 + c0 + 2 * e, sq.len, p.causal, p.window)) a = 0.f;
                if (!allowed(il, j0 + c0 + 2 * e + 1, sq.len, p.causal, p.window)) b = 0.f;
              }
              pk[e] = pack2<BF16>(a, b);
            }
            tmem_st16(tS + c0 / 2, pk);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive_warp(&ctl.p_full[u & 1]);
          mbar_arrive_warp(&ctl.s_free[buf]);
        }
      }
      if (n == 0) lse2 = (l > 0.f) ? mx + log2f(l) : INFINITY;
      // epilogue: O (already normalised) and LSE
      if (ok && mbar_wait_warp(&ctl.acc_done, 0, guard, 7)) {
        tc_fence_after();
        const bool valid = il < sq.len;
        const size_t orow = (static_cast<size_t>(zq) * p.S + sq.start + il);
        T* o = static_cast<T*>(out) + orow * DV;
#pragma unroll 1
        for (int c0 = 0; c0 < DV; c0 += 32) {
          uint32_t v[32];
          if (n > 0) tmem_ld32(tmem + lane_base + C::T_ACC + c0, v);
          else
            for (int e = 0; e < 32; ++e) v[e] = 0u;
          if (valid) {
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint4 w;
              w.x = pack2<BF16>(__uint_as_float(v[8 * q4 + 0]), __uint_as_float(v[8 * q4 + 1]));
              w.y = pack2<BF16>(__uint_as_float(v[8 * q4 + 2]), __uint_as_float(v[8 * q4 + 3]));
              w.z = pack2<BF16>(__uint_as_float(v[8 * q4 + 4]), __uint_as_float(v[8 * q4 + 5]));
              w.w = pack2<BF16>(__uint_as_float(v[8 * q4 + 6]), __uint_as_float(v[8 * q4 + 7]));
              *reinterpret_cast<uint4*>(o + c0 + 8 * q4) = w;
            }
          }
        }
        if (valid) lse_out[orow] = lse2 * kLn2;
      }
    } else {
      // deterministic dQ pass
      const size_t sidx = stat_index(p, h, s, t) + r;
      const float nlse2 = p.nlse2[sidx];
      const float ndlt = p.ndelta[sidx];
      for (int it = 0; it < NIT; ++it) {
        const int kt = k0 + it;
        const int j0 = kt * C::BK;
        const bool need_mask = (j0 + C::BK > sq.len) || (p.causal && j0 + C::BK - 1 > t * C::BQ) ||
                               (p.window > 0 && t * C::BQ + C::BQ - 1 - j0 >= p.window);
        if (!mbar_wait_warp(&ctl.s_full[0], it & 1, guard, 6)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tS = tmem + lane_base + C::T_S0, tP = tmem + lane_base + C::T_S1;
#pragma unroll 1
        for (int c0 = 0; c0 < C::BK; c0 += 32) {
          uint32_t sv[32], dv[32];
          tmem_ld32(tS + c0, sv);
          tmem_ld32(tP + c0, dv);
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float pa = ex2_approx(fmaf(__uint_as_float(sv[2 * e]), sl2, nlse2));
            float pb = ex2_approx(fmaf(__uint_as_float(sv[2 * e + 1]), sl2, nlse2));
            if (need_mask) {
              if (!allowed(il, j0 + c0 + 2 * e, sq.len, p.causal, p.window)) pa = 0.f;
              if (!allowed(il, j0 + c0 + 2 * e + 1, sq.len, p.causal, p.window)) pb = 0.f;
            }
            const float da = pa * (__uint_as_float(dv[2 * e]) + ndlt);
            const float db = pb * (__uint_as_float(dv[2 * e + 1]) + ndlt);
            pk[e] = pack2<BF16>(da, db);
          }
          tmem_st16(tP + c0 / 2, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(&ctl.p_full[0]);
        mbar_arrive_warp(&ctl.s_free[0]);
      }
      if (ok && mbar_wait_warp(&ctl.acc_done, 0, guard, 7)) {
        tc_fence_after();
        const bool valid = il < sq.len;
        const size_t qrow = static_cast<size_t>(zq) * p.S + sq.start + il;
        T* dq = static_cast<T*>(out) + qrow * DQK;
        if (n > 0) {
#pragma unroll 1
          for (int c0 = 0; c0 < DQK; c0 += 32) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_base + C::T_ACC + c0, v);  // all lanes: .sync.aligned
            if (!valid) continue;
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint4 w;
              w.x = pack2<BF16>(__uint_as_float(v[8 * q4 + 0]) * p.scale, __uint_as_float(v[8 * q4 + 1]) * p.scale);
              w.y = pack2<BF16>(__uint_as_float(v[8 * q4 + 2]) * p.scale, __uint_as_float(v[8 * q4 + 3]) * p.scale);
              w.z = pack2<BF16>(__uint_as_float(v[8 * q4 + 4]) * p.scale, __uint_as_float(v[8 * q4 + 5]) * p.scale);
              w.w = pack2<BF16>(__uint_as_float(v[8 * q4 + 6]) * p.scale, __uint_as_float(v[8 * q4 + 7]) * p.scale);
              *reinterpret_cast<uint4*>(dq + c0 + 8 * q4) = w;
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
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

cudaError_t launch_fwd(const Problem& p, int dtype_bf16, const Maps& m, const float* sink, void* o, float* lse,
                       cudaStream_t st) {
  return dispatch_q<true>(p, dtype_bf16, m, sink, o, lse, st);
}

cudaError_t launch_dq(const Problem& p, int dtype_bf16, const Maps& m, void* dq, cudaStream_t st) {
  return dispatch_q<false>(p, dtype_bf16, m, nullptr, dq, nullptr, st);
}

}  // namespace gqa
