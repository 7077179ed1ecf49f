// Query-stationary tcgen05 dQ pass: one CTA owns 128 query rows of one query
// head and streams the 64-row key/value tiles they can see.  Per key tile it
// recomputes S = Q.K^T and dP = dO.V^T, forms dS = P*(dP - Delta) with
// P = exp2(S*scale*log2e - LSE2) (tilelang-ascend PR #1638 "Add GQA Sink Backward
// BHSD", review thread k1..k5, in the loop order the Ascend kernel uses for dQ,
// "dQ[L0C accumulate]"), and accumulates dQ += dS.K in TMEM with no atomics;
// dQ * scale is written once.  It serves the deterministic mode (bit-identical
// run to run) and the dQ of head dim 192, whose key-stationary main kernel has
// no TMEM room for a dQ accumulator.
//
// Warp roles (320 threads): warps 0-3 and 4-7 are two softmax warpgroups that
// take alternate key tiles (warpgroup w the tiles with index parity w), thread r
// owns query row r = TMEM lane r; warp 8 = TMA producer; warp 9 = TMEM allocator
// + MMA issuer (the whole warp runs the loop, one lane elected per MMA).  Tile
// `it` has the TMEM buffer it % 2: while one warpgroup works on its tile the
// tensor core computes the other's.  Operands live in shared memory in the
// 128-byte swizzled layout TMA writes; S, dP and dQ accumulate in TMEM; dS is
// packed to 16 bits over S and feeds the dQ MMA as its A operand.  The
// stationary dO tile (and Q, where the TMEM columns allow) is copied into TMEM
// once and is the A operand of dP (and S).
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <type_traits>
#include "common.cuh"
#include "umma.cuh"
#include "launch.h"

namespace gqa {

template <int DQK, int DV>
struct QCfg {
  static constexpr int BQ = 128;  // query rows = TMEM lanes
  static constexpr int BK = 64;   // keys per tile
  static constexpr int Q_BYTES = BQ * DQK * 2;
  static constexpr int DO_BYTES = BQ * DV * 2;
  static constexpr int K_BYTES = BK * DQK * 2;
  static constexpr int V_BYTES = BK * DV * 2;
  static constexpr int STAGE_BYTES = K_BYTES + V_BYTES;  // one K + V stage
  // the dO tile is read once, by the softmax warps that copy it into TMEM: it is loaded into the last
  // K/V stage, which takes its first key tile only after that copy (one more stage in flight)
  static constexpr int BUDGET = 220 * 1024;
  static constexpr int KST_RAW = (BUDGET - Q_BYTES) / STAGE_BYTES;
  static constexpr int KST = KST_RAW > 8 ? 8 : KST_RAW;
  static constexpr int SMEM = 1024 + Q_BYTES + KST * STAGE_BYTES;
  // TMEM: buffer b at b*BUF holds S (BK columns; dS packed over its first half) and dP right after
  // it; the dQ accumulator follows the two buffers
  static constexpr int NBUF = 2;
  static constexpr uint32_t BUF = 2 * BK;
  static constexpr uint32_t T_ACC = NBUF * BUF;
  // the stationary dO and Q tiles as TMEM A operands (packed 16-bit pairs, like P), after the
  // accumulator: dO always, Q where the 512 columns allow (head dims 64 and 128).  The N = 64 S and dP
  // MMAs then read only their B operand (the key tile) from shared memory: with both operands there
  // they need 6 KB per 32 cycles of math, more than shared memory's 128 bytes per cycle
  static constexpr uint32_t T_DO = T_ACC + DQK;
  static constexpr uint32_t T_Q = T_DO + DV / 2;
  static constexpr bool Q_TMEM = T_Q + DQK / 2 <= 512;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr int THREADS = 320;
  static_assert(KST >= 2, "stages");
  static_assert(DO_BYTES <= STAGE_BYTES, "the dO tile fits in one K/V stage");
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(T_DO + DV / 2 <= 512, "tmem");
  static_assert(DQK % 64 == 0, "each warpgroup drains whole 32-column chunks");
};

struct QSmemCtl {
  uint64_t bar_q;
  uint64_t kv_full[8], kv_empty[8];
  uint64_t s_full[2];   // tensor core -> warpgroup: S and dP of the buffer's tile are in TMEM
  uint64_t sm_done[2];  // warpgroup -> tensor core: dS stored, buffer reusable
  uint64_t acc_done;
  uint64_t op_tmem;     // softmax warps -> tensor core and producer: dO (and Q) copied into TMEM
  uint32_t tmem_base;
  int abort_flag;
};

template <int DQK, int DV, bool BF16>
__global__ void __launch_bounds__(320, 1)
    q_kernel(const Problem p, const __grid_constant__ Maps m, void* __restrict__ out) {
  using C = QCfg<DQK, DV>;
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  extern __shared__ uint8_t smem_raw[];
  __shared__ QSmemCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sK0 = sQ + C::Q_BYTES;  // stage st: K at sK0 + st*STAGE_BYTES, V right after K
  uint8_t* sDO = sK0 + (C::KST - 1) * C::STAGE_BYTES;  // until it is in TMEM

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
  const int NIT = k1 - k0;
  const int g = h / p.G;
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
    for (int i = 0; i < C::NBUF; ++i) {
      mbar_init(&ctl.s_full[i], 1);
      mbar_init(&ctl.sm_done[i], 4);  // one arrival per warp of the warpgroup
    }
    mbar_init(&ctl.acc_done, 1);
    mbar_init(&ctl.op_tmem, 8);  // one arrival per softmax warp
    ctl.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(&ctl.tmem_base, C::TMEM_COLS);
    tmem_relinquish();
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
      for (int cb = 0; cb < DQK / 64; ++cb) tma_load_4d(sQ + cb * (C::BQ * 128), &m.q, &ctl.bar_q, cb * 64, row0, h, sq.b);
      for (int cb = 0; cb < DV / 64; ++cb)
        tma_load_4d(sDO + cb * (C::BQ * 128), &m.dout, &ctl.bar_q, cb * 64, row0, h, sq.b);
      int issued = 0;
      for (int it = 0; it < NIT; ++it) {
        const int st = it % C::KST;
        if (it >= C::KST && !mbar_wait(&ctl.kv_empty[st], ((it / C::KST) - 1) & 1, guard, 1)) break;
        // the last stage holds dO until the softmax warps have copied it into TMEM
        if (it == C::KST - 1 && !mbar_wait(&ctl.op_tmem, 0, guard, 10)) break;
        uint8_t* sK = sK0 + st * C::STAGE_BYTES;
        uint8_t* sV = sK + C::K_BYTES;
        mbar_expect_tx(&ctl.kv_full[st], C::K_BYTES + C::V_BYTES);
        const int krow = sk.start + (k0 + it) * C::BK;
        for (int cb = 0; cb < DQK / 64; ++cb)
          tma_load_4d(sK + cb * (C::BK * 128), &m.k, &ctl.kv_full[st], cb * 64, krow, g, sk.b);
        for (int cb = 0; cb < DV / 64; ++cb)
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
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    {  // the whole warp runs the issue loop; one elected lane issues each MMA
      constexpr uint32_t idS = idesc_f16(128, C::BK, BF16, false, false);
      constexpr uint32_t idDQ = idesc_f16(128, DQK, BF16, false, true);
      const uint64_t dQ0 = sdesc_sw128(smem_u32(sQ), 16, 1024);    // Q, K-major (A of S)
      auto kstep = [](int kk, int rows) -> uint32_t { return (kk / 4) * (rows * 128) + (kk % 4) * 32; };
      bool ok = mbar_wait_warp(&ctl.bar_q, 0, guard, 2);
      if (ok && NIT > 0) ok = mbar_wait_warp(&ctl.op_tmem, 0, guard, 9);
      // S and dP of tile `it` into buffer it % 2, once the tile two earlier has left it
      // `waited`: the caller has already waited for the K/V tile and for the buffer's previous tile
      auto issue_s = [&](int it, bool waited) -> bool {
        const int st = it % C::KST, b = it % C::NBUF;
        if (!waited) {
          if (!mbar_wait_warp(&ctl.kv_full[st], (it / C::KST) & 1, guard, 3)) return false;
          if (it >= C::NBUF && !mbar_wait_warp(&ctl.sm_done[b], ((it - C::NBUF) / C::NBUF) & 1, guard, 4))
            return false;
        }
        tc_fence_after();
        const uint32_t aK = smem_u32(sK0 + st * C::STAGE_BYTES);
        const uint64_t dK = sdesc_sw128(aK, 16, 1024);
        const uint64_t dV = sdesc_sw128(aK + C::K_BYTES, 16, 1024);
        const uint32_t tS = tmem + b * C::BUF;
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk) {
          if constexpr (C::Q_TMEM)
            umma_ts(tS, tmem + C::T_Q + kk * 8, desc_advance(dK, kstep(kk, C::BK)), idS, kk > 0);
          else
            umma_ss(tS, desc_advance(dQ0, kstep(kk, C::BQ)), desc_advance(dK, kstep(kk, C::BK)), idS, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk)
          umma_ts(tS + C::BK, tmem + C::T_DO + kk * 8, desc_advance(dV, kstep(kk, C::BK)), idS, kk > 0);
        umma_commit(&ctl.s_full[b]);
        return true;
      };
      // dQ += dS.K -- A = the packed dS in the tile's buffer, B = K read MN-major
      auto issue_acc = [&](int it) -> bool {
        const int st = it % C::KST, b = it % C::NBUF;
        if (!mbar_wait_warp(&ctl.sm_done[b], (it / C::NBUF) & 1, guard, 5)) return false;
        tc_fence_after();
        const uint64_t dKmn = sdesc_sw128(smem_u32(sK0 + st * C::STAGE_BYTES), C::BK * 128, 1024);
        const uint32_t tA = tmem + b * C::BUF;
#pragma unroll
        for (int kk = 0; kk < C::BK / 16; ++kk)
          umma_ts(tmem + C::T_ACC, tA + kk * 8, desc_advance(dKmn, kk * 2048), idDQ, (it > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&ctl.kv_empty[st]);
        return true;
      };
      for (int it = 0; ok && it < C::NBUF && it < NIT; ++it) ok = issue_s(it, false);
      // in the order the warpgroups release the buffers: tile it's accumulation, then the
      // tile that takes its buffer next (the accumulation's wait for tile it is also the wait for the
      // buffer).  With a deep K/V ring the next tile's K/V wait comes first, while the softmax still
      // works on tile it; with a shallow one that load may still be in flight, and the accumulation
      // goes first.
      constexpr bool EARLY_KV = C::KST >= 6;
      for (int it = 0; ok && it < NIT; ++it) {
        const int nx = it + C::NBUF;
        const bool more = nx < NIT;
        if (EARLY_KV && more && !mbar_wait_warp(&ctl.kv_full[nx % C::KST], (nx / C::KST) & 1, guard, 3)) break;
        if (!issue_acc(it)) break;
        if (!EARLY_KV && more && !mbar_wait_warp(&ctl.kv_full[nx % C::KST], (nx / C::KST) & 1, guard, 3)) break;
        if (more && !issue_s(nx, true)) break;
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
    bool ok = true;
    const size_t sidx = stat_index(p, h, s, t) + r;
    const float nlse2 = p.nlse2[sidx];
    const float ndlt = p.ndelta[sidx];
    // warpgroup 0 copies dO, warpgroup 1 Q (where it goes to TMEM) into TMEM: thread r moves row r,
    // 128 bytes per 64-column block (128-byte swizzled in shared memory: 16-byte chunk c of row r sits
    // at chunk c ^ (r % 8)) into 32 packed columns of lane r
    if (NIT > 0) {
      if (!mbar_wait_warp(&ctl.bar_q, 0, guard, 8)) {
        ok = false;
      } else {
        if (w == 0 || C::Q_TMEM) {
          const uint8_t* base = (w == 0) ? sDO : sQ;
          const int ncb = (w == 0) ? DV / 64 : DQK / 64;
          const uint32_t tdst = tmem + lane_base + ((w == 0) ? C::T_DO : C::T_Q);
#pragma unroll 1
          for (int cb = 0; cb < ncb; ++cb) {
            const uint8_t* row = base + cb * (C::BQ * 128) + r * 128;
            uint32_t wd[2][16];
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint4 u = *reinterpret_cast<const uint4*>(row + ((c ^ (r & 7)) * 16));
              wd[c / 4][(c % 4) * 4 + 0] = u.x;
              wd[c / 4][(c % 4) * 4 + 1] = u.y;
              wd[c / 4][(c % 4) * 4 + 2] = u.z;
              wd[c / 4][(c % 4) * 4 + 3] = u.w;
            }
            tmem_st16(tdst + cb * 32, wd[0]);
            tmem_st16(tdst + cb * 32 + 16, wd[1]);
          }
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive_warp(&ctl.op_tmem);
      }
    }
    for (int it = w; ok && it < NIT; it += 2) {
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
      const float2 sl22 = make_float2(sl2, sl2), nl2 = make_float2(nlse2, nlse2), nd2 = make_float2(ndlt, ndlt);
      // dS of the 32 key columns starting at c0 from their S and dP, packed over S's first half: chunk
      // c0 lands in columns [c0/2, c0/2 + 16), which earlier chunks have already read
      auto ds_chunk = [&](int c0, const uint32_t (&sv)[32], const uint32_t (&dv)[32]) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          // P = exp2(S * scale * log2e - LSE2) and dS = P * (dP - Delta), two columns at a time
          const float2 x = fma2(make_float2(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), sl22, nl2);
          const float2 pp = make_float2(ex2_approx(x.x), ex2_approx(x.y));
          const float2 d = mul2(pp, add2(make_float2(__uint_as_float(dv[2 * e]), __uint_as_float(dv[2 * e + 1])), nd2));
          pk[e] = pack2<BF16>(d.x, d.y);
        }
        // masked keys: dS = P * (dP - Delta) is 0 where P is, so their packed halves are cleared (one test
        // per chunk on the unmasked tiles)
        if (need_mask) {
          const int d0 = il + off - j0 - c0;  // diagonal distance to this chunk's first key
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (!visible_d(d0 - e, j0 + c0 + e < sk.len, p.right, p.window)) pk[e / 2] &= (e & 1) ? 0x0000FFFFu : 0xFFFF0000u;
        }
        tmem_st16(tS + c0 / 2, pk);
      };
      // the two 32-column chunks of the tile: the second one's S and dP load while the first is used
      static_assert(C::BK == 64, "two 32-column chunks");
      uint32_t s0[32], d0v[32], s1[32], d1v[32];
      tmem_ld32_start(tS, s0);
      tmem_ld32_start(tS + C::BK, d0v);
      tmem_ld_wait(s0);
      tmem_ld_wait(d0v);
      tmem_ld32_start(tS + 32, s1);
      tmem_ld32_start(tS + C::BK + 32, d1v);
      ds_chunk(0, s0, d0v);
      tmem_ld_wait(s1);
      tmem_ld_wait(d1v);
      ds_chunk(32, s1, d1v);
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
        if (NIT > 0) tmem_ld32(tmem + lane_base + C::T_ACC + c0, v);  // all lanes: .sync.aligned
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

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int DQK, int DV, bool BF16>
static cudaError_t launch_q_t(const Problem& p, const Maps& m, void* out, cudaStream_t st) {
  using C = QCfg<DQK, DV>;
  auto kern = q_kernel<DQK, DV, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int ntiles = (p.max_len + C::BQ - 1) / C::BQ;
  if (ntiles == 0 || p.nseqs == 0) return cudaSuccess;
  dim3 grid(p.Hq, ntiles, p.nseqs);
  kern<<<grid, C::THREADS, C::SMEM, st>>>(p, m, out);
  return cudaGetLastError();
}

cudaError_t launch_dq(const Problem& p, int dtype_bf16, const Maps& m, void* dq, cudaStream_t st) {
#define GQA_Q(DQK, DV)                                                                                      \
  if (p.Dqk == DQK && p.Dv == DV)                                                                           \
    return dtype_bf16 ? launch_q_t<DQK, DV, true>(p, m, dq, st) : launch_q_t<DQK, DV, false>(p, m, dq, st);
  GQA_Q(64, 64)
  GQA_Q(128, 128)
  GQA_Q(192, 128)
#undef GQA_Q
  return cudaErrorInvalidValue;
}

int q_kernel_bk() { return QCfg<64, 64>::BK; }

}  // namespace gqa
