// Key/value-stationary tcgen05 backward main kernel.
//
// One CTA owns 128 key/value rows (one KV tile) of one kv head and streams the
// query tiles that can see them (tilelang PR #1093 "[GQA] Add regional atomic
// add", Additional comments: per-KV-block CTAs, a k_base loop over query blocks,
// dQ added per iteration, dK/dV accumulated locally and added once into kv head
// "bx // groups").  Per query tile it computes (tilelang-ascend PR #1638 "Add GQA
// Sink Backward BHSD", review thread k1..k5), transposed so the 128 key rows
// sit on the 128 TMEM lanes:
//
//   S^T  = K . Q^T                (tcgen05, fp32 in TMEM)
//   P^T  = exp2(S^T*scale*log2e - LSE2_i), masked      (CUDA cores, packed to 16-bit in TMEM)
//   dP^T = V . dO^T               (tcgen05)
//   dS^T = P^T * (dP^T - Delta_i) (CUDA cores; 16-bit in TMEM and, for dQ, in shared memory)
//   dV  += P^T . dO               (tcgen05, A operand from TMEM)
//   dK  += dS^T . Q               (tcgen05, A operand from TMEM)
//   dQ_partial = dS . K           (tcgen05) -> added into an fp32 dQ accumulator
//
// The softmax scale is left out of dS and applied once to dK (epilogue) and dQ
// (postprocess).  Group reduction of dK/dV over the Hq/Hkv query heads:
//   group_tmem = 1 : the CTA loops over every query head of its kv head, so dK/dV
//                    stay in TMEM and are written once as fp16/bf16 (no atomics);
//   group_tmem = 0 : one CTA per query head; after its loop it adds dK/dV into
//                    fp32 accumulators (red.v4 / bulk tensor reduce / scalar red).
// dQ partials are added with red.global.add.v4.f32, a bulk tensor reduce from
// shared memory (cp.reduce.async.bulk.tensor), or per-element red.f32 (triton
// issue #4717 "atomic_add slows down attention backwards due to layout
// conversions": vectorised atomics against scalar ones).
//
// For head dim 64 the stationary K and V tiles are also copied into TMEM and
// serve as the A operands of S^T and dP^T, and dS^T is packed over dP^T.
//
// Warp roles (448 threads): warps 0-3 and 4-7 are two softmax/dS warpgroups
// (thread r = key row r = TMEM lane r; the first takes query columns [0, BQ/2),
// the second [BQ/2, BQ)); warps 8-11 dQ drain warpgroup (thread r = query row r);
// warp 12 TMA producer; warp 13 TMEM allocator + MMA issuer.
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <type_traits>
#include "common.cuh"
#include "umma.cuh"
#include "launch.h"

namespace gqa {

template <int DQK, int DV>
struct KvCfg {
  static constexpr int BK = 128;
  static constexpr int BQ = (DQK == 64) ? 128 : 64;      // query rows per tile
  static constexpr bool HAS_DQ = (DQK != 192);          // (192,128): dQ from the query-stationary pass
  // d=128: dQ^T = K^T . dS^T with the head dim on the 128 TMEM lanes (a 64-row query tile cannot
  // be the M of an MMA); the tile is transposed through shared memory for the reduction
  static constexpr bool DQ_T = (DQK == 128);
  static constexpr bool HAS_STAGING = (DQK == 64);       // per-warp 32x32 staging for the bulk dQ reduce
  static constexpr int K_BYTES = BK * DQK * 2, V_BYTES = BK * DV * 2;
  static constexpr int Q_BYTES = BQ * DQK * 2, DO_BYTES = BQ * DV * 2;
  static constexpr int ST = 3;
  static constexpr int DS_BYTES = HAS_DQ ? BQ * BK * 2 : 0;   // one dS tile; two alternate
  // head dim 64: -LSE/scale and -Delta enter Sᵀ and dPᵀ through one extra K=16 MMA each (an xfold
  // tile of bf16 hi + mid + lo terms per stage against constant ones operands) instead of
  // per-element shared-memory loads
  static constexpr bool FOLD = (DQK == 64);
  static constexpr int X_BYTES = FOLD ? BQ * kFoldRowBytes : 0;
  static constexpr int STAT_BYTES = FOLD ? 0 : BQ * 4;          // LSE / Delta vector per stage
  static constexpr int STG_BYTES = HAS_STAGING ? 4 * 32 * 32 * 4 : (DQ_T ? BQ * DQK * 4 : 0);
  // shared-memory map (offsets from a 1024-aligned base)
  static constexpr int OFF_K = 0, OFF_V = OFF_K + K_BYTES;
  static constexpr int OFF_Q = OFF_V + V_BYTES;                  // stage st at OFF_Q + st*Q_BYTES
  static constexpr int OFF_DO = OFF_Q + ST * Q_BYTES;
  static constexpr int OFF_DS = OFF_DO + ST * DO_BYTES;
  static constexpr int OFF_STG = OFF_DS + 2 * DS_BYTES;
  static constexpr int OFF_LSE = OFF_STG + STG_BYTES;           // ST x BQ floats (not FOLD)
  static constexpr int OFF_DEL = OFF_LSE + ST * STAT_BYTES;
  static constexpr int OFF_X = OFF_DEL + ST * STAT_BYTES;        // ST xfold tiles (FOLD)
  static constexpr int OFF_ONES = OFF_X + ST * X_BYTES;          // FOLD: 3 core matrices ones|zeros|ones
  static constexpr int ONES_BYTES = FOLD ? 384 : 0;
  static constexpr int OFF_CTL = OFF_ONES + ONES_BYTES;
  static constexpr int SMEM = OFF_CTL + 256;
  // TMEM columns
  static constexpr uint32_t T_S = 0, T_DP = BQ, T_DV = 2 * BQ, T_DK = 2 * BQ + DV;
  static constexpr uint32_t T_DQ = T_DK + DQK;  // dQ (DQK cols) or dQ^T (BQ cols)
  // packed dS^T (BQ/2 columns) in the 64 columns every head-dim configuration leaves free, so the
  // next tile's dP^T can be computed while dK still reads this tile's dS^T
  static constexpr uint32_t T_DSP = 448;
  // head dim 64: the stationary K and V tiles are also copied into TMEM (the last 64 columns, packed
  // 16-bit like P), so S^T = K . Q^T and dP^T = V . dO^T take their A operand from TMEM instead of
  // shared memory (32 KB less shared-memory traffic per tile); packed dS^T then goes over dP^T, like
  // P^T over S^T, and the next tile's dP^T follows this tile's dK
  static constexpr bool KV_TMEM = (DQK == 64 && DV == 64);
  static constexpr uint32_t T_K = 448, T_V = 480;
  static constexpr int HALF = BQ / 2;                   // query columns per softmax warpgroup
  static constexpr int NCH = HALF / 32;                   // 32-column chunks per softmax warpgroup
  static constexpr int THREADS = 448;
  static_assert(SMEM <= 232448, "shared memory");
  static_assert(T_DK + DQK <= T_DSP && (!HAS_DQ || T_DQ + (DQ_T ? BQ : DQK) <= T_DSP), "tmem");
  static_assert(T_DSP + BQ / 2 <= 512, "tmem");
  static_assert(!KV_TMEM || (T_DQ + DQK <= T_K && T_V + DV / 2 <= 512 && BQ == 128), "tmem: K and V");
  // the dK/dV epilogue stages bulk reductions in the idle Q/dO stage buffers (8 warps x 8 KB)
  static_assert(ST * (Q_BYTES + DO_BYTES) >= 8 * 2 * 32 * 32 * 4, "epilogue staging");
};

struct KvCtl {
  uint64_t kv_full;
  uint64_t q_full[3], do_full[3], q_empty[3];
  uint64_t s_full, dp_full, p_full, ds_full, ds_free;
  uint64_t dq_full, dq_empty, dsmem_free[2], acc_done;
  uint64_t kv_tmem;  // K and V copied into TMEM (head dim 64)
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(KvCtl) <= 256, "ctl");


__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* m, const void* src, int c0, int c1, int c2) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// Same box as tma_reduce_add_3d, plain store (the no-accumulation benchmark mode).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* m, const void* src, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(m)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void bulk_wait_read1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

// Adds a warp's 32 rows x 32 fp32 columns (one row per lane, in v[]) into a
// global fp32 accumulator, by the chosen mode.  `grow` = global row of this lane
// (row of [rows][ld]), `valid` = lane's row is inside its sequence.
template <int MODE>
__device__ __forceinline__ void add_row32(float* acc, size_t grow, int ld, int c0, const uint32_t (&v)[32],
                                          bool valid) {
  if (!valid) return;
  float* dst = acc + grow * ld + c0;
  if (MODE == kDqRedV4) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      red_add_v4(dst + 4 * q, __uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                 __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
  } else if (MODE == kDqScalar) {
#pragma unroll
    for (int e = 0; e < 32; ++e) red_add_f32(dst + e, __uint_as_float(v[e]));
  } else if (MODE == kDqStore) {
#pragma unroll
    for (int q = 0; q < 8; ++q)
      *reinterpret_cast<float4*>(dst + 4 * q) = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                                            __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
  }
}

// Bulk path: stage a warp's 32x32 fp32 block in 128B-swizzled shared memory
// (the layout the fp32 reduce tensor map expects) and reduce it with one TMA op.
__device__ __forceinline__ void stage_and_reduce(uint8_t* stg, const CUtensorMap* map, int lane, const uint32_t (&v)[32],
                                                 int x, int y, int z, bool store = false) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint32_t off = lane * 128 + ((q ^ (lane & 7)) * 16);
    *reinterpret_cast<uint4*>(stg + off) = make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  }
  fence_async_smem();
  __syncwarp();
  if (lane == 0) {
    if (store) tma_store_3d(map, stg, x, y, z);
    else tma_reduce_add_3d(map, stg, x, y, z);
    bulk_commit();
  }
}

// One TMEM load of a warpgroup's half of the query columns (32 or 64 columns).
template <int N>
__device__ __forceinline__ void tmem_ld_half(uint32_t taddr, uint32_t (&v)[N]);
template <>
__device__ __forceinline__ void tmem_ld_half<64>(uint32_t taddr, uint32_t (&v)[64]) {
  tmem_ld64(taddr, v);
}
template <>
__device__ __forceinline__ void tmem_ld_half<32>(uint32_t taddr, uint32_t (&v)[32]) {
  tmem_ld32(taddr, v);
}

template <int DQK, int DV, bool BF16>
__global__ void __launch_bounds__(448, 1)
    kv_kernel(const Problem p, const __grid_constant__ Maps m, const int group_tmem, const int dq_mode,
              const int kv_mode, void* __restrict__ dk_out, void* __restrict__ dv_out) {
  using C = KvCfg<DQK, DV>;
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  extern __shared__ __align__(1024) uint8_t smem[];
  KvCtl& ctl = *reinterpret_cast<KvCtl*>(smem + C::OFF_CTL);

  const int head = blockIdx.x;   // kv head (group_tmem) or query head
  // y = KV tile (tile 0 has the most query tiles under a causal mask: launched first); z = sequence
  // slot, mapped to a sequence by the longest-first order of packed batches
  const int s = p.sched ? p.sched[blockIdx.z] : static_cast<int>(blockIdx.z);
  if (static_cast<unsigned>(s) >= static_cast<unsigned>(p.nseqs)) {  // no preprocess on this workspace
    if (threadIdx.x == 0) atomicCAS(p.err, 0, kErrBadSeqlens);
    return;
  }
  Seq sq, sk;  // the sequence's queries and keys
  if (!load_seq(p, s, sq) || !load_kseq(p, s, sk)) return;
  const int off = sk.len - sq.len;  // query i sits on key diagonal i + off
  const int ntk = (sk.len + C::BK - 1) / C::BK;
  const int kt = blockIdx.y;
  if (kt >= ntk) return;
  if ((smem_u32(smem) & 1023u) != 0) {  // the operand layout needs a 1024-byte aligned base
    if (threadIdx.x == 0) atomicCAS(p.err, 0, 0x40000010);
    return;
  }
  int t0, t1;
  q_tiles_for_kv_tile(kt, sq.len, sk.len, C::BQ, p.right, p.window, &t0, &t1);
  const int nt = t1 - t0;
  const int g = group_tmem ? head : head / p.G;
  const int nh = group_tmem ? p.G : 1;
  const int h_first = group_tmem ? g * p.G : head;
  const int NIT = nh * nt;
  const int j0 = kt * C::BK;
  const int zk = sq.b * p.Hkv + g;

  // the warp index goes through a shuffle so the compiler knows it is warp-uniform: the warp-role
  // branches below are then uniform and the MMA operands can stay in uniform registers
  const int tid = threadIdx.x, warp = __shfl_sync(0xffffffffu, tid >> 5, 0), lane = tid & 31;
  if (tid == 0) {
    mbar_init(&ctl.kv_full, 1);
    for (int i = 0; i < C::ST; ++i) {
      mbar_init(&ctl.q_full[i], 1);
      mbar_init(&ctl.do_full[i], 1);
      mbar_init(&ctl.q_empty[i], 1);
    }
    mbar_init(&ctl.s_full, 1);
    mbar_init(&ctl.dp_full, 1);
    mbar_init(&ctl.p_full, 8);   // one arrival per softmax warp
    mbar_init(&ctl.ds_full, 8);
    mbar_init(&ctl.ds_free, 1);
    mbar_init(&ctl.dq_full, 1);
    mbar_init(&ctl.dq_empty, 4);  // one arrival per drain warp
    mbar_init(&ctl.dsmem_free[0], 1);
    mbar_init(&ctl.dsmem_free[1], 1);
    mbar_init(&ctl.acc_done, 1);
    mbar_init(&ctl.kv_tmem, 8);  // one arrival per softmax warp
    ctl.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 13) {
    tmem_alloc(&ctl.tmem_base, 512);
    tmem_relinquish();
  }
  if (C::FOLD && tid < C::ONES_BYTES / 16) {
    // bf16 core matrices ones | zeros | ones: the A operands that add the xfold columns 0-7
    // (start 0) or 8-15 (start 128) of each query row to every logit of that row
    const uint32_t v = (tid / 8 == 1) ? 0u : 0x3F803F80u;
    reinterpret_cast<uint4*>(smem + C::OFF_ONES)[tid] = make_uint4(v, v, v, v);
    fence_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // broadcast from lane 0 so the compiler treats the TMEM base as warp-uniform (uniform registers
  // for the MMA operands instead of per-MMA register moves)
  const uint32_t tmem = __shfl_sync(0xffffffffu, ctl.tmem_base, 0);
  const WaitGuard guard{p.err, &ctl.abort_flag, p.wait_limit};

  if (warp == 12) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_map(&m.q);
      tma_prefetch_map(&m.dout);
      mbar_expect_tx(&ctl.kv_full, C::K_BYTES + C::V_BYTES);
      const int krow = sk.start + j0;
      for (int cb = 0; cb < DQK / 64; ++cb)
        tma_load_4d(smem + C::OFF_K + cb * (C::BK * 128), &m.k, &ctl.kv_full, cb * 64, krow, g, sk.b);
      for (int cb = 0; cb < DV / 64; ++cb)
        tma_load_4d(smem + C::OFF_V + cb * (C::BK * 128), &m.v, &ctl.kv_full, cb * 64, krow, g, sk.b);
      int issued = 0;
      for (int it = 0; it < NIT; ++it) {
        const int st = it % C::ST;
        if (it >= C::ST && !mbar_wait(&ctl.q_empty[st], ((it / C::ST) - 1) & 1, guard, 11)) break;
        const int h = h_first + it / nt;
        const int t = t0 + it % nt;
        const int qrow = sq.start + t * C::BQ;
        uint8_t* sQ = smem + C::OFF_Q + st * C::Q_BYTES;
        uint8_t* sDO = smem + C::OFF_DO + st * C::DO_BYTES;
        const size_t sidx = stat_index(p, h, s, (t * C::BQ) / kStatTile) + (t * C::BQ) % kStatTile;
        mbar_expect_tx(&ctl.q_full[st], C::Q_BYTES + (C::FOLD ? C::X_BYTES : 2 * C::STAT_BYTES));
        for (int cb = 0; cb < DQK / 64; ++cb)
          tma_load_4d(sQ + cb * (C::BQ * 128), &m.q, &ctl.q_full[st], cb * 64, qrow, h, sq.b);
        if (C::FOLD) {
          // the tile's rows are contiguous in the xfold layout (whole 8-row groups)
          bulk_load(smem + C::OFF_X + st * C::X_BYTES, p.xfold + sidx * kFoldRowBytes, C::X_BYTES, &ctl.q_full[st]);
        } else {
          bulk_load(smem + C::OFF_LSE + st * C::STAT_BYTES, p.nlse2 + sidx, C::STAT_BYTES, &ctl.q_full[st]);
          bulk_load(smem + C::OFF_DEL + st * C::STAT_BYTES, p.ndelta + sidx, C::STAT_BYTES, &ctl.q_full[st]);
        }
        mbar_expect_tx(&ctl.do_full[st], C::DO_BYTES);
        for (int cb = 0; cb < DV / 64; ++cb)
          tma_load_4d(sDO + cb * (C::BQ * 128), &m.dout, &ctl.do_full[st], cb * 64, qrow, h, sq.b);
        issued = it + 1;
      }
      if (ctl.abort_flag) {
        volatile int no_abort = 0;
        const WaitGuard g2{nullptr, &no_abort, p.wait_limit};
        mbar_wait(&ctl.kv_full, 0, g2, 0);
        for (int it = issued - C::ST < 0 ? 0 : issued - C::ST; it < issued; ++it) {
          mbar_wait(&ctl.q_full[it % C::ST], (it / C::ST) & 1, g2, 0);
          mbar_wait(&ctl.do_full[it % C::ST], (it / C::ST) & 1, g2, 0);
        }
      }
    }
  } else if (warp == 13) {
    // ------------------------------------------------------------ MMA issuer
    {  // the whole warp runs the issue loop; one elected lane issues each MMA
      constexpr uint32_t idS = idesc_f16(128, C::BQ, BF16, false, false);
      constexpr uint32_t idDV = idesc_f16(128, DV, BF16, false, true);
      constexpr uint32_t idDK = idesc_f16(128, DQK, BF16, false, true);
      // d=64: dQ = dS . K (M = query rows); d=128: dQ^T = K^T . dS^T (M = head dim)
      constexpr uint32_t idDQ = C::DQ_T ? idesc_f16(128, C::BQ, BF16, true, true)
                                        : idesc_f16(C::BQ, (DQK <= 256 ? DQK : 256), BF16, true, true);
      const bool dq_on = C::HAS_DQ && dq_mode != kDqNone;
      // packed 16-bit P^T / dS^T: each softmax warpgroup packs its half of the query
      // columns into the first half of its own column range
      auto a_col = [](int kk) -> uint32_t {
        return static_cast<uint32_t>((kk / (C::HALF / 16)) * C::HALF + (kk % (C::HALF / 16)) * 8);
      };
      // shared-memory descriptors, built once and advanced by compile-time offsets
      const uint64_t dK_k = sdesc_sw128(smem_u32(smem + C::OFF_K), 16, 1024);          // K tile, K-major
      const uint64_t dK_mn = sdesc_sw128(smem_u32(smem + C::OFF_K), C::BK * 128, 1024); // K tile, MN-major
      const uint64_t dV_k = sdesc_sw128(smem_u32(smem + C::OFF_V), 16, 1024);
      const uint64_t dDS_mn = sdesc_sw128(smem_u32(smem + C::OFF_DS), C::BK * 128, 1024);
      const uint64_t dQ_k0 = sdesc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
      const uint64_t dQ_mn0 = sdesc_sw128(smem_u32(smem + C::OFF_Q), C::BQ * 128, 1024);
      const uint64_t dDO_k0 = sdesc_sw128(smem_u32(smem + C::OFF_DO), 16, 1024);
      const uint64_t dDO_mn0 = sdesc_sw128(smem_u32(smem + C::OFF_DO), C::BQ * 128, 1024);
      // the fold: ones (A, bf16, no swizzle, one core matrix pair for every row group) x xfold tile (B, bf16)
      constexpr uint32_t idF = idesc_f16(128, C::BQ, true, false, false);
      const uint64_t dAL = sdesc_none(smem_u32(smem + C::OFF_ONES), 128, 0);        // K columns 0-7
      const uint64_t dAD = sdesc_none(smem_u32(smem + C::OFF_ONES) + 128, 128, 0);  // K columns 8-15
      const uint64_t dX0 = sdesc_none(smem_u32(smem + C::OFF_X), 128, 256);
      // K-major operand with 64-element (128-byte) rows: K step kk lives in 64-column block kk/4 at byte kk%4*32
      auto kstep = [](int kk, int rows) -> uint32_t { return (kk / 4) * (rows * 128) + (kk % 4) * 32; };
      bool ok = mbar_wait_warp(&ctl.kv_full, 0, guard, 12);
      if (C::KV_TMEM && ok && NIT > 0) ok = mbar_wait_warp(&ctl.kv_tmem, 0, guard, 26);
      auto issue_s = [&](int it) -> bool {
        const int st = it % C::ST;
        if (!mbar_wait_warp(&ctl.q_full[st], (it / C::ST) & 1, guard, 13)) return false;
        tc_fence_after();
        const uint64_t dq = desc_advance(dQ_k0, st * C::Q_BYTES);
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk) {
          if constexpr (C::KV_TMEM)
            umma_ts(tmem + C::T_S, tmem + C::T_K + kk * 8, desc_advance(dq, kstep(kk, C::BQ)), idS, kk > 0);
          else
            umma_ss(tmem + C::T_S, desc_advance(dK_k, kstep(kk, C::BK)), desc_advance(dq, kstep(kk, C::BQ)), idS, kk > 0);
        }
        if (C::FOLD) umma_ss(tmem + C::T_S, dAL, desc_advance(dX0, st * C::X_BYTES), idF, 1u);  // - LSE/scale
        umma_commit(&ctl.s_full);
        return true;
      };
      auto issue_dp = [&](int it) -> bool {
        const int st = it % C::ST;
        if (!mbar_wait_warp(&ctl.do_full[st], (it / C::ST) & 1, guard, 14)) return false;
        tc_fence_after();
        const uint64_t ddo = desc_advance(dDO_k0, st * C::DO_BYTES);
#pragma unroll
        for (int kk = 0; kk < DV / 16; ++kk) {
          if constexpr (C::KV_TMEM)
            umma_ts(tmem + C::T_DP, tmem + C::T_V + kk * 8, desc_advance(ddo, kstep(kk, C::BQ)), idS, kk > 0);
          else
            umma_ss(tmem + C::T_DP, desc_advance(dV_k, kstep(kk, C::BK)), desc_advance(ddo, kstep(kk, C::BQ)), idS, kk > 0);
        }
        if (C::FOLD) umma_ss(tmem + C::T_DP, dAD, desc_advance(dX0, st * C::X_BYTES), idF, 1u);  // - Delta
        umma_commit(&ctl.dp_full);
        return true;
      };
      if (ok && NIT > 0) ok = issue_s(0) && issue_dp(0);
      for (int it = 0; ok && it < NIT; ++it) {
        const int st = it % C::ST;
        const uint64_t dq_mn = desc_advance(dQ_mn0, st * C::Q_BYTES);
        const uint64_t ddo_mn = desc_advance(dDO_mn0, st * C::DO_BYTES);
        // dV += P^T . dO
        if (!mbar_wait_warp(&ctl.p_full, it & 1, guard, 16)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < C::BQ / 16; ++kk)
          umma_ts(tmem + C::T_DV, tmem + C::T_S + a_col(kk), desc_advance(ddo_mn, kk * 2048), idDV,
                  (it > 0 || kk > 0) ? 1u : 0u);
        // next tile's S^T (its columns were read by the softmax warps, P^T was consumed by the dV MMA above)
        if (it + 1 < NIT && !issue_s(it + 1)) break;
        if (!mbar_wait_warp(&ctl.ds_full, it & 1, guard, 17)) break;
        if constexpr (C::KV_TMEM) {
          // dK += dS^T . Q with dS^T packed over dP^T, then the next tile's dP^T over the same columns
          // (tcgen05.mma runs in issue order, so dK has read dS^T before dP^T overwrites it)
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < C::BQ / 16; ++kk)
            umma_ts(tmem + C::T_DK, tmem + C::T_DP + a_col(kk), desc_advance(dq_mn, kk * 2048), idDK,
                    (it > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&ctl.ds_free);
          umma_commit(&ctl.q_empty[st]);
          if (it + 1 < NIT && !issue_dp(it + 1)) break;
        } else {
          // the softmax warps are idle until the next tile's dP^T: it goes first, then dK += dS^T . Q
          if (it + 1 < NIT && !issue_dp(it + 1)) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < C::BQ / 16; ++kk)
            umma_ts(tmem + C::T_DK, tmem + C::T_DSP + kk * 8, desc_advance(dq_mn, kk * 2048), idDK,
                    (it > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&ctl.ds_free);
          // the Q / dO stage is free once dK has read Q (S^T, dP^T and dV read it earlier): the producer
          // loads the tile ST ahead while the dQ MMAs below, which read K and dS only, still run
          umma_commit(&ctl.q_empty[st]);
        }
        // dQ_partial = dS . K
        if (dq_on) {
          if (it >= 1 && !mbar_wait_warp(&ctl.dq_empty, (it - 1) & 1, guard, 18)) break;
          tc_fence_after();
          const uint32_t ds_off = (it & 1) * C::DS_BYTES;  // dS tiles alternate between two buffers
          if (C::DQ_T) {
            // dQ^T = K^T . dS^T : A = K tile read MN-major, B = dS read MN-major (query contiguous)
#pragma unroll
            for (int kk = 0; kk < C::BK / 16; ++kk)
              umma_ss(tmem + C::T_DQ, desc_advance(dK_mn, kk * 2048), desc_advance(dDS_mn, ds_off + kk * 2048), idDQ, kk > 0);
          } else {
            // dQ = dS . K : A = dS read MN-major (query contiguous), B = K tile read MN-major
#pragma unroll
            for (int kk = 0; kk < C::BK / 16; ++kk)
              umma_ss(tmem + C::T_DQ, desc_advance(dDS_mn, ds_off + kk * 2048), desc_advance(dK_mn, kk * 2048), idDQ, kk > 0);
          }
          umma_commit(&ctl.dq_full);
          umma_commit(&ctl.dsmem_free[it & 1]);
        }
      }
      umma_commit(&ctl.acc_done);
    }
  } else if (warp >= 8) {
    // ------------------------------------------------------------ dQ drain warpgroup
    if (C::HAS_DQ && dq_mode != kDqNone) {
      const int r = tid - 256;  // query row within the tile == TMEM lane
      const uint32_t lane_base = static_cast<uint32_t>((warp - 8) * 32) << 16;
      uint8_t* stg = smem + C::OFF_STG + (warp - 8) * (32 * 32 * 4);
      int nbulk = 0;
      for (int it = 0; it < NIT; ++it) {
        const int h = h_first + it / nt;
        const int t = t0 + it % nt;
        const int il = t * C::BQ + r;
        bool got = mbar_wait_warp(&ctl.dq_full, it & 1, guard, 19);
        // the transposing path meets at named barriers below: the four drain warps decide together
        // whether to go on, so none leaves the loop while a sibling waits at a barrier for it
        if (C::DQ_T) got = named_bar_and(2, 128, got);
        if (!got) break;
        tc_fence_after();
        if (C::DQ_T) {
          // thread r = head-dim column r: the tile is transposed through shared memory
          float* tst = reinterpret_cast<float*>(smem + C::OFF_STG);  // [BQ query rows][DQK]
          uint32_t v[C::BQ];
          tmem_ld_half<C::BQ>(tmem + lane_base + C::T_DQ, v);
          tc_fence_before();
          mbar_arrive_warp(&ctl.dq_empty);
          const int row0 = t * C::BQ;
          const int nvalid = sq.len - row0 < C::BQ ? sq.len - row0 : C::BQ;
          float* gdst = p.dq_acc + ((static_cast<size_t>(sq.b) * p.Hq + h) * p.S + sq.start + row0) * DQK;
          if (dq_mode == kDqBulk || dq_mode == kDqStore) {  // kDqStore: the same copies, stored
            // two halves of BQ/2 query rows, each staged in its own half of the buffer and reduced by its
            // own bulk operation: a half is written while the other half's previous reduce still reads
            // shared memory, instead of every tile waiting for the whole previous reduce
            constexpr int HQ = C::BQ / 2;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              float* hst = tst + hh * HQ * DQK;
              // one bulk group per half (empty when the half has no valid row): the group two back read
              // this half of the buffer
              if (r == 0 && nbulk >= 2) bulk_wait_read1();
              named_bar_sync(1, 128);
#pragma unroll
              for (int i = 0; i < HQ; ++i) hst[i * DQK + r] = __uint_as_float(v[hh * HQ + i]);
              fence_async_smem();
              named_bar_sync(1, 128);
              const int nv = nvalid - hh * HQ < 0 ? 0 : (nvalid - hh * HQ > HQ ? HQ : nvalid - hh * HQ);
              if (r == 0) {  // the half's rows are contiguous in the accumulator
                if (nv > 0) {
                  if (dq_mode == kDqStore) bulk_store_f32(gdst + hh * HQ * DQK, hst, static_cast<uint32_t>(nv) * DQK * 4);
                  else bulk_reduce_add_f32(gdst + hh * HQ * DQK, hst, static_cast<uint32_t>(nv) * DQK * 4);
                }
                bulk_commit();
              }
              ++nbulk;
            }
          } else {
            named_bar_sync(1, 128);
#pragma unroll
            for (int i = 0; i < C::BQ; ++i) tst[i * DQK + r] = __uint_as_float(v[i]);
            named_bar_sync(1, 128);
            const float4* s4 = reinterpret_cast<const float4*>(tst);
            for (int idx = r; idx < nvalid * (DQK / 4); idx += 128) {
              const float4 x = s4[idx];
              float* dst = gdst + 4 * idx;
              if (dq_mode == kDqRedV4) {
                red_add_v4(dst, x.x, x.y, x.z, x.w);
              } else if (dq_mode == kDqScalar) {
                red_add_f32(dst, x.x);
                red_add_f32(dst + 1, x.y);
                red_add_f32(dst + 2, x.z);
                red_add_f32(dst + 3, x.w);
              } else {
                *reinterpret_cast<float4*>(dst) = x;
              }
            }
            named_bar_sync(1, 128);  // staging free for the next tile
          }
          continue;
        }
        if constexpr (C::HAS_STAGING) {
          if (dq_mode == kDqBulk || dq_mode == kDqStore) {  // kDqStore: same copies, stored
            // the whole row into registers, release the accumulator, then stage and reduce each
            // 32-column chunk through this warp's single staging buffer
            uint32_t v[DQK];
            tmem_ld_half<DQK>(tmem + lane_base + C::T_DQ, v);
            tc_fence_before();
            mbar_arrive_warp(&ctl.dq_empty);
#pragma unroll
            for (int c = 0; c < DQK / 32; ++c) {
              uint32_t w[32];
#pragma unroll
              for (int e = 0; e < 32; ++e) w[e] = v[32 * c + e];
              if (lane == 0 && nbulk >= 1) bulk_wait_read0();  // the previous reduce has read the buffer
              __syncwarp();
              stage_and_reduce(stg, &m.dq_acc, lane, w, 32 * c, sq.start + t * C::BQ + (warp - 8) * 32,
                               sq.b * p.Hq + h, dq_mode == kDqStore);
              ++nbulk;
            }
            continue;
          }
        }
        const size_t grow = (static_cast<size_t>(sq.b) * p.Hq + h) * p.S + sq.start + il;
        const bool valid = il < sq.len;
#pragma unroll
        for (int c = 0; c < DQK / 32; ++c) {
          const int c0 = 32 * c;
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + C::T_DQ + c0, v);
          if (c == DQK / 32 - 1) {  // every column is in registers: release the accumulator
            tc_fence_before();
            mbar_arrive_warp(&ctl.dq_empty);
          }
          if (dq_mode == kDqRedV4) add_row32<kDqRedV4>(p.dq_acc, grow, DQK, c0, v, valid);
          else if (dq_mode == kDqScalar) add_row32<kDqScalar>(p.dq_acc, grow, DQK, c0, v, valid);
          else if (dq_mode == kDqStore) add_row32<kDqStore>(p.dq_acc, grow, DQK, c0, v, valid);
        }
      }
      if (nbulk > 0 && (C::DQ_T ? r == 0 : lane == 0)) bulk_wait0();
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ softmax / dS warpgroups
    const int wg = warp >> 2;          // which half of the query columns
    const int r = tid & 127;           // key row within the tile == TMEM lane
    const int j = j0 + r;
    const int cbase = wg * C::HALF;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
    const bool dq_on = C::HAS_DQ && dq_mode != kDqNone;
    bool ok = true;
    if constexpr (C::KV_TMEM) {
      // warpgroup 0 copies K, warpgroup 1 V into TMEM: thread r moves key row r (128 bytes, 128-byte
      // swizzled in shared memory: 16-byte chunk c of row r sits at chunk c ^ (r % 8)) into 32 packed
      // columns of lane r
      if (NIT > 0) {
        if (!mbar_wait_warp(&ctl.kv_full, 0, guard, 27)) {
          ok = false;
        } else {
          const uint8_t* row = smem + (wg == 0 ? C::OFF_K : C::OFF_V) + r * 128;
          uint32_t w[2][16];
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 u = *reinterpret_cast<const uint4*>(row + ((c ^ (r & 7)) * 16));
            w[c / 4][(c % 4) * 4 + 0] = u.x;
            w[c / 4][(c % 4) * 4 + 1] = u.y;
            w[c / 4][(c % 4) * 4 + 2] = u.z;
            w[c / 4][(c % 4) * 4 + 3] = u.w;
          }
          const uint32_t tkv = tmem + lane_base + (wg == 0 ? C::T_K : C::T_V);
          tmem_st16(tkv, w[0]);
          tmem_st16(tkv + 16, w[1]);
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive_warp(&ctl.kv_tmem);
        }
      }
    }
    for (int it = 0; ok && it < NIT; ++it) {
      const int st = it % C::ST;
      const int t = t0 + it % nt;
      const int i0 = t * C::BQ;
      const bool need_mask = (j0 + C::BK > sk.len) || (p.right > 0 && i0 + off + p.right < j0 + C::BK) ||
                             (p.window > 0 && i0 + C::BQ - 1 + off - j0 >= p.window);
      const float4* sL4 = reinterpret_cast<const float4*>(smem + C::OFF_LSE) + (st * C::BQ + cbase) / 4;
      const float4* sD4 = reinterpret_cast<const float4*>(smem + C::OFF_DEL) + (st * C::BQ + cbase) / 4;
      // exponent arguments of four consecutive columns: S*scale*log2e - LSE2 (with the fold the MMA
      // already subtracted LSE/scale, so only the scaling remains)
      auto exp_args = [&](const uint32_t* v4, const float4* l4, float2 s2, float2& x0, float2& x1) {
        const float2 a = make_float2(__uint_as_float(v4[0]), __uint_as_float(v4[1]));
        const float2 b = make_float2(__uint_as_float(v4[2]), __uint_as_float(v4[3]));
        if constexpr (C::FOLD) {
          x0 = mul2(a, s2);
          x1 = mul2(b, s2);
        } else {
          const float4 l = *l4;
          x0 = fma2(a, s2, make_float2(l.x, l.y));
          x1 = fma2(b, s2, make_float2(l.z, l.w));
        }
      };
      if (!mbar_wait_warp(&ctl.q_full[st], (it / C::ST) & 1, guard, 20) ||
          !mbar_wait_warp(&ctl.s_full, it & 1, guard, 21)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // P^T = exp2(S^T * scale*log2e - LSE2) for this warpgroup's columns, kept packed (16-bit) for dS
      uint32_t pk[C::HALF / 2];
      auto p_chunk = [&](int c, const uint32_t (&v)[32]) {
        if (BF16) {
          float pf[32];
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            float2 x0, x1;
            exp_args(v + 4 * q4, sL4 + 8 * c + q4, sl2, x0, x1);
            pf[4 * q4 + 0] = ex2_approx(x0.x);
            pf[4 * q4 + 1] = ex2_approx(x0.y);
            pf[4 * q4 + 2] = ex2_approx(x1.x);
            pf[4 * q4 + 3] = ex2_approx(x1.y);
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) pk[16 * c + e] = pack2<true>(pf[2 * e], pf[2 * e + 1]);
        } else {
          // fp16: the exponent argument is rounded to fp16 and exponentiated two at a time; the
          // result is the packed P the MMA consumes (argument rounding adds at most ~2e-4 to P)
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4) {
            float2 x0, x1;
            exp_args(v + 4 * q4, sL4 + 8 * c + q4, sl2, x0, x1);
            pk[16 * c + 2 * q4] = ex2_f16x2(pack2<false>(x0.x, x0.y));
            pk[16 * c + 2 * q4 + 1] = ex2_f16x2(pack2<false>(x1.x, x1.y));
          }
        }
        if (need_mask) {
          const int d0 = i0 + cbase + 32 * c + off - j;  // diagonal distance of this chunk's first query
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (!visible_d(d0 + e, j < sk.len, p.right, p.window)) pk[16 * c + e / 2] &= (e & 1) ? 0x0000FFFFu : 0xFFFF0000u;
        }
        uint32_t pc[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pc[e] = pk[16 * c + e];
        tmem_st16(tmem + lane_base + C::T_S + cbase + 16 * c, pc);
      };
      // 32-column chunks: the second one's load runs while the first is exponentiated
      {
        uint32_t va[32];
        tmem_ld32(tmem + lane_base + C::T_S + cbase, va);
        if constexpr (C::NCH == 2) {
          uint32_t vb[32];
          tmem_ld32_start(tmem + lane_base + C::T_S + cbase + 32, vb);
          p_chunk(0, va);
          tmem_ld_wait(vb);
          p_chunk(1, vb);
        } else {
          p_chunk(0, va);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(&ctl.p_full);
      // dS^T = P^T * (dP^T - Delta): the difference in fp32, the product on packed 16-bit pairs
      if (!mbar_wait_warp(&ctl.dp_full, it & 1, guard, 22)) {
        ok = false;
        break;
      }
      if (dq_on && it >= 2 && !mbar_wait_warp(&ctl.dsmem_free[it & 1], ((it - 2) >> 1) & 1, guard, 23)) {
        ok = false;
        break;
      }
      // the previous tile's dK MMA must have read its dS^T before this one is stored
      if (it >= 1 && !mbar_wait_warp(&ctl.ds_free, (it - 1) & 1, guard, 25)) {
        ok = false;
        break;
      }
      tc_fence_after();
      auto ds_chunk = [&](int c, const uint32_t (&v)[32]) {
        uint32_t ds[16];
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          float2 a = make_float2(__uint_as_float(v[4 * q4]), __uint_as_float(v[4 * q4 + 1]));
          float2 b = make_float2(__uint_as_float(v[4 * q4 + 2]), __uint_as_float(v[4 * q4 + 3]));
          if constexpr (!C::FOLD) {  // with the fold the MMA already subtracted Delta
            const float4 d = sD4[8 * c + q4];
            a = add2(a, make_float2(d.x, d.y));
            b = add2(b, make_float2(d.z, d.w));
          }
          ds[2 * q4] = mul_packed<BF16>(pk[16 * c + 2 * q4], pack2<BF16>(a.x, a.y));
          ds[2 * q4 + 1] = mul_packed<BF16>(pk[16 * c + 2 * q4 + 1], pack2<BF16>(b.x, b.y));
        }
        tmem_st16(tmem + lane_base + (C::KV_TMEM ? C::T_DP + cbase : C::T_DSP + cbase / 2) + 16 * c, ds);
        if (dq_on) {
          // dS for the dQ MMA: MN-major (query index contiguous), 128B swizzle, key row r = K index
          const int c0 = cbase + 32 * c;
          uint8_t* sds = smem + C::OFF_DS + (it & 1) * C::DS_BYTES + (c0 / 64) * (C::BK * 128) + r * 128;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int chunk = ((c0 % 64) / 8 + q) ^ (r & 7);
            *reinterpret_cast<uint4*>(sds + chunk * 16) = make_uint4(ds[4 * q], ds[4 * q + 1], ds[4 * q + 2], ds[4 * q + 3]);
          }
        }
      };
      {
        uint32_t va[32];
        tmem_ld32(tmem + lane_base + C::T_DP + cbase, va);
        if constexpr (C::NCH == 2) {
          // the second chunk's dP^T is read before the first chunk's dS^T is stored over dP^T's columns
          // 0-15 of this warpgroup (and it never overlaps them: its columns are 32-63)
          uint32_t vb[32];
          tmem_ld32_start(tmem + lane_base + C::T_DP + cbase + 32, vb);
          ds_chunk(0, va);
          tmem_ld_wait(vb);
          ds_chunk(1, vb);
        } else {
          ds_chunk(0, va);
        }
      }
      tmem_st_wait();
      if (dq_on) fence_async_smem();
      tc_fence_before();
      mbar_arrive_warp(&ctl.ds_full);
    }
    // ---------------------------------------------------------- dK / dV epilogue
    // warpgroup 0 writes dV, warpgroup 1 writes dK (both cover all 128 key rows)
    if (ok && mbar_wait_warp(&ctl.acc_done, 0, guard, 24)) {
      tc_fence_after();
      const bool valid = j < sk.len;
      const size_t krow = static_cast<size_t>(zk) * p.Sk + sk.start + j;
      uint8_t* stg = smem + C::OFF_Q + warp * (2 * 32 * 32 * 4);  // stage buffers are idle now
      int nbulk = 0;
      auto emit = [&](uint32_t tcol, int D, void* out, const Strides& ost, float* acc, const CUtensorMap* map,
                      float mul) {
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t v[32];
          if (NIT > 0) tmem_ld32(tmem + lane_base + tcol + c0, v);
          else
            for (int e = 0; e < 32; ++e) v[e] = 0u;
          if (group_tmem) {
            if (valid) {
              T* o = static_cast<T*>(out) + ost.row(sk.b, g, sk.start + j) + c0;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                uint4 w;
                w.x = pack2<BF16>(__uint_as_float(v[8 * q + 0]) * mul, __uint_as_float(v[8 * q + 1]) * mul);
                w.y = pack2<BF16>(__uint_as_float(v[8 * q + 2]) * mul, __uint_as_float(v[8 * q + 3]) * mul);
                w.z = pack2<BF16>(__uint_as_float(v[8 * q + 4]) * mul, __uint_as_float(v[8 * q + 5]) * mul);
                w.w = pack2<BF16>(__uint_as_float(v[8 * q + 6]) * mul, __uint_as_float(v[8 * q + 7]) * mul);
                *reinterpret_cast<uint4*>(o + 8 * q) = w;
              }
            }
          } else if (kv_mode == kDqRedV4) {
            add_row32<kDqRedV4>(acc, krow, D, c0, v, valid);
          } else if (kv_mode == kDqScalar) {
            add_row32<kDqScalar>(acc, krow, D, c0, v, valid);
          } else if (kv_mode == kDqStore) {
            add_row32<kDqStore>(acc, krow, D, c0, v, valid);
          } else {
            uint8_t* buf = stg + (nbulk & 1) * (32 * 32 * 4);
            if (lane == 0 && nbulk >= 1) bulk_wait_read1();
            __syncwarp();
            stage_and_reduce(buf, map, lane, v, c0, sk.start + j0 + (warp & 3) * 32, zk);
            ++nbulk;
          }
        }
      };
      if (wg == 0) emit(C::T_DV, DV, dv_out, p.dv_st, p.dv_acc, &m.dv_acc, 1.f);
      else emit(C::T_DK, DQK, dk_out, p.dk_st, p.dk_acc, &m.dk_acc, p.scale);
      if (lane == 0 && nbulk > 0) bulk_wait0();
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DQK, int DV, bool BF16>
static cudaError_t launch_kv_t(const Problem& p, const Maps& m, const KvLaunch& kl, cudaStream_t st) {
  using C = KvCfg<DQK, DV>;
  auto kern = kv_kernel<DQK, DV, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int ntk = (p.max_len_k + C::BK - 1) / C::BK;
  if (ntk == 0 || p.nseqs == 0) return cudaSuccess;
  dim3 grid(kl.group_tmem ? p.Hkv : p.Hq, ntk, p.nseqs);
  kern<<<grid, C::THREADS, C::SMEM, st>>>(p, m, kl.group_tmem, C::HAS_DQ ? kl.dq_mode : kDqNone, kl.kv_red_mode,
                                          kl.dk, kl.dv);
  return cudaGetLastError();
}

cudaError_t launch_bwd_kv(const Problem& p, int dtype_bf16, const Maps& m, const KvLaunch& kl, cudaStream_t st) {
#define GQA_KV(DQK, DV)                                                                            \
  if (p.Dqk == DQK && p.Dv == DV)                                                                  \
    return dtype_bf16 ? launch_kv_t<DQK, DV, true>(p, m, kl, st) : launch_kv_t<DQK, DV, false>(p, m, kl, st);
  GQA_KV(64, 64)
  GQA_KV(128, 128)
  GQA_KV(192, 128)
#undef GQA_KV
  return cudaErrorInvalidValue;
}

bool kv_kernel_has_dq(int Dqk) { return Dqk != 192; }
bool kv_kernel_folds_stats(int Dqk) { return Dqk == 64; }
bool kv_kernel_has_bulk_dq(int Dqk) { return Dqk != 192; }
int kv_kernel_bq(int Dqk) { return Dqk == 64 ? 128 : 64; }

}  // namespace gqa
