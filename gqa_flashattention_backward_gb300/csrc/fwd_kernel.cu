// One-pass tcgen05 forward with causal / sliding-window / attention-sink masking
// (tilelang-ascend PR #1638 "Add GQA Sink Backward BHSD", 4->2 commit:
// "flashattn_fwd: online softmax + sink + window -> O, lse").
//
// One CTA owns two 128-row query tiles of one query head; softmax warpgroup w
// (warps 4w..4w+3, thread r = query row r of tile w = TMEM lane r) keeps its own
// running row maximum, row sum and O accumulator, so the two tiles need no
// exchange and take turns on the tensor core.  The CTA loads every key tile
// either query tile can see; with 128-key tiles each warpgroup (and the MMA
// warp on its behalf) skips the tiles that its own rows cannot see (a sliding
// window's far edge, the other tile's causal diagonal).  Per key tile of BK keys:
//
//   S_w  = Q_w . K^T                     (tcgen05, fp32 in TMEM)
//   m_ref = reference maximum of S_w * scale * log2(e) (below)
//   P_w  = exp2(S_w * scale * log2(e) - m_ref), packed to 16 bits into TMEM
//   O_w += P_w . V                        (tcgen05, A operand from TMEM)
//
// The softmax reads its whole S row into registers with one TMEM load and one
// wait, and works on it in code compiled twice: with the causal / window /
// length mask (the tiles on a diagonal or an edge) and without.  For head dim
// 64 P has TMEM columns of its own, so S_w of the next key tile is computed as
// soon as the row is read, while this tile's exponentials run; the softmax waits
// for P_w . V of the previous tile only before it writes P and O.  For head dims
// 128 (S and O fill the 512 columns) and 192 P is packed over S and the next S
// follows this tile's P.V.
//
// m_ref, the maximum P is taken against, starts at the sink or at the first
// tile's maximum and moves only when a tile's row sum of P -- which bounds each
// of its P -- exceeds 2^TAU; then the warp rescales its O rows in TMEM (and the
// row sums) by exp2(m_ref_old - m_ref_new) and recomputes P from the registers.
// No per-element maximum is taken.  O = O_w / l and LSE = ln 2 * (m_ref + log2 l).
//
// Warp roles (384 threads): warps 0-3 / 4-7 the two softmax warpgroups (240
// registers each after the launch's 168 are redistributed), warp 8 the TMA
// producer of the Q tiles and the K ring, warp 10 that of the V ring, warp 9 the
// TMEM allocator and MMA issuer (whole warp, one lane elected per MMA), warp 11
// idle (its registers go to the softmax).
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <type_traits>
#include "common.cuh"
#include "fwd_tiles.cuh"
#include "umma.cuh"
#include "launch.h"

namespace gqa {

template <int DQK, int DV, bool BF16>
struct FwdCfg {
  static constexpr int BQ = 128;                     // query rows per warpgroup tile = TMEM lanes
  static constexpr int BK = (DQK <= 128) ? 128 : 64;  // keys per tile
  static constexpr int Q_BYTES = BQ * DQK * 2;        // one query tile
  static constexpr int K_BYTES = BK * DQK * 2, V_BYTES = BK * DV * 2;
  static constexpr int BUDGET = 225 * 1024;
  // K stages first (S runs ahead of P.V), then V stages
  static constexpr int VST = 2;
  static constexpr int KST_RAW = (BUDGET - 2 * Q_BYTES - VST * V_BYTES) / K_BYTES;
  static constexpr int KST = KST_RAW > 4 ? 4 : KST_RAW;
  static constexpr int SMEM = 1024 + 2 * Q_BYTES + KST * K_BYTES + VST * V_BYTES;
  // TMEM per warpgroup: S (BK columns) then O (DV columns).  For head dim 64 P has columns of its own
  // (BK/2 packed per warpgroup, after both warpgroups' S and O): S of the next key tile is then
  // computed as soon as the softmax has read S, while P.V of this tile still reads P.  Otherwise P is
  // packed over S, which the next S waits for (head dim 128: S and O fill the 512 columns; head dim
  // 192: its 64-key S tiles are short, and the tensor core rather than the softmax sets the pace).
  static constexpr uint32_t WG_COLS = BK + DV;
  static constexpr bool SEP_P = DQK == 64;
  // each warpgroup on its own key tiles only (128-key tiles).  With 64-key tiles (head dim 192) the MMA
  // warp issues an S MMA every ~32 cycles and sets the pace, and the per-tile range tests cost more
  // than the two masked tiles per pair they save: both warpgroups then run the union
  static constexpr bool OWN_RANGES = BK == 128;
  static constexpr uint32_t P_COL = 2 * WG_COLS;  // SEP_P: P of warpgroup w at P_COL + w * BK / 2
  static constexpr uint32_t TMEM_COLS = 512;
  // P <= 2^TAU: m_ref moves only when a tile's row sum of P exceeds P_MAX = 2^TAU.  fp16 exponentiates
  // the argument rounded to fp16 (relative error of P at most 2^-9 ln 2 for arguments up to TAU) and
  // adds 32 values of P at most 2^TAU each in fp16 (at most 2^13: far inside its range)
  static constexpr float TAU = 8.f, P_MAX = 256.f;
  // 12 warps (three per SM sub-partition: 168 registers each at launch); the softmax warpgroups take
  // 240 registers (a whole S row stays in registers), the TMA / MMA warpgroup keeps 24
  static constexpr int THREADS = 384;
  static constexpr uint32_t SOFTMAX_REGS = 240, OTHER_REGS = 24;
  static_assert(8 * 32 * SOFTMAX_REGS + 4 * 32 * OTHER_REGS <= 168 * THREADS, "register split");
  static_assert(KST >= 2, "key stages");
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(2 * WG_COLS + (SEP_P ? BK : 0) <= TMEM_COLS, "tmem");
  static_assert(BK == 64 || BK == 128, "S row load");
  static_assert(BK % 32 == 0 && DV % 64 == 0, "chunks");
};

__device__ __forceinline__ __half2 u32_as_half2(uint32_t x) {
  __half2 r;
  memcpy(&r, &x, sizeof(r));
  return r;
}

struct FwdCtl {
  uint64_t bar_q;
  uint64_t k_full[4], k_empty[4];
  uint64_t v_full[2], v_empty[2];
  uint64_t s_full[2];   // tensor core -> warpgroup w: S_w of the next key tile is in TMEM
  uint64_t s_free[2];   // warpgroup w -> tensor core: S_w read into registers (separate P only)
  uint64_t p_full[2];   // warpgroup w -> tensor core: P_w stored (O_w rescaled)
  uint64_t pv_done[2];  // tensor core -> warpgroup w: P_w . V of the last tile done (separate P only)
  uint64_t acc_done;
  uint32_t tmem_base;
  int abort_flag;
};

template <int DQK, int DV, bool BF16>
__global__ void __launch_bounds__(384, 1)
    fwd_kernel(const Problem p, const __grid_constant__ Maps m, const float* __restrict__ sink, void* __restrict__ out,
               float* __restrict__ lse_out) {
  using C = FwdCfg<DQK, DV, BF16>;
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  extern __shared__ uint8_t smem_raw[];
  __shared__ FwdCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                          // tile w at sQ + w * Q_BYTES
  uint8_t* sK0 = sQ + 2 * C::Q_BYTES;          // K stage st at sK0 + st * K_BYTES
  uint8_t* sV0 = sK0 + C::KST * C::K_BYTES;    // V stage st at sV0 + st * V_BYTES

  const int h = blockIdx.x;
  const int s = blockIdx.z;
  Seq sq, sk;
  if (!load_seq(p, s, sq) || !load_kseq(p, s, sk)) return;
  const int off = sk.len - sq.len;  // query i sits on key diagonal i + off
  const int npair = (sq.len + 2 * C::BQ - 1) / (2 * C::BQ);
  const int tp = static_cast<int>(gridDim.y) - 1 - static_cast<int>(blockIdx.y);  // heavy tile pairs first
  if (tp >= npair) return;
  // the union [k0, k0 + n) of the two query tiles' key tiles, which the CTA loads; with OWN_RANGES
  // warpgroup w works (and the MMA warp issues for it) only on its own tiles, local indices
  // jlo_w <= j < jhi_w of the union, otherwise both on all n (scalars, so that no runtime index puts
  // them in local memory)
  int k0, n, jlo0, jhi0, jlo1, jhi1;
  fwd_pair_tiles(tp, sq.len, sk.len, C::BK, p.right, p.window, &k0, &n, &jlo0, &jhi0, &jlo1, &jhi1);
  if constexpr (!C::OWN_RANGES) {
    jlo0 = jlo1 = 0;
    jhi0 = jhi1 = n;
  }
  const int g = h / p.G;
  const int zq = sq.b * p.Hq + h;

  const int tid = threadIdx.x, warp = __shfl_sync(0xffffffffu, tid >> 5, 0), lane = tid & 31;
  if (tid == 0) {
    mbar_init(&ctl.bar_q, 1);
    for (int i = 0; i < C::KST; ++i) {
      mbar_init(&ctl.k_full[i], 1);
      mbar_init(&ctl.k_empty[i], 1);
    }
    for (int i = 0; i < C::VST; ++i) {
      mbar_init(&ctl.v_full[i], 1);
      mbar_init(&ctl.v_empty[i], 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(&ctl.s_full[w], 1);
      mbar_init(&ctl.s_free[w], 4);  // one arrival per warp of the warpgroup
      mbar_init(&ctl.p_full[w], 4);
      mbar_init(&ctl.pv_done[w], 1);
    }
    mbar_init(&ctl.acc_done, 1);
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
  const uint32_t tmem = __shfl_sync(0xffffffffu, ctl.tmem_base, 0);
  const WaitGuard guard{p.err, &ctl.abort_flag, p.wait_limit};

  if (warp >= 8) {
    reg_dealloc<C::OTHER_REGS>();
    if (warp == 8 || warp == 10) {
      // ------------------------------------------------------------ TMA producers: warp 8 the Q tiles
      // and the K ring, warp 10 the V ring, so that neither ring waits for a slot of the other
      if (lane == 0) {
        const bool is_k = warp == 8;
        const CUtensorMap* map = is_k ? &m.k : &m.v;
        uint64_t* full = is_k ? ctl.k_full : ctl.v_full;
        uint64_t* empty = is_k ? ctl.k_empty : ctl.v_empty;
        const int nst = is_k ? C::KST : C::VST;
        const int bytes = is_k ? C::K_BYTES : C::V_BYTES;
        const int cbs = is_k ? DQK / 64 : DV / 64;
        uint8_t* base = is_k ? sK0 : sV0;
        tma_prefetch_map(map);
        if (is_k) {
          tma_prefetch_map(&m.q);
          mbar_expect_tx(&ctl.bar_q, 2 * C::Q_BYTES);
          for (int w = 0; w < 2; ++w)
            for (int cb = 0; cb < DQK / 64; ++cb)
              tma_load_4d(sQ + w * C::Q_BYTES + cb * (C::BQ * 128), &m.q, &ctl.bar_q, cb * 64,
                          sq.start + (2 * tp + w) * C::BQ, h, sq.b);
        }
        int issued = 0;
        for (int i = 0; i < n; ++i) {
          const int st = i % nst;
          if (i >= nst && !mbar_wait(&empty[st], ((i / nst) - 1) & 1, guard, 1)) break;
          mbar_expect_tx(&full[st], bytes);
          for (int cb = 0; cb < cbs; ++cb)
            tma_load_4d(base + st * bytes + cb * (C::BK * 128), map, &full[st], cb * 64, sk.start + (k0 + i) * C::BK,
                        g, sk.b);
          issued = i + 1;
        }
        // the last copies of the ring have landed before the CTA's shared memory can go away (also when
        // another warp gave up on a wait and the tiles are never consumed)
        volatile int no_abort = 0;
        const WaitGuard g2{nullptr, &no_abort, p.wait_limit};
        if (is_k) mbar_wait(&ctl.bar_q, 0, g2, 0);
        for (int i = issued - nst < 0 ? 0 : issued - nst; i < issued; ++i)
          mbar_wait(&full[i % nst], (i / nst) & 1, g2, 0);
      }
    } else if (warp == 9) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idS = idesc_f16(128, C::BK, BF16, false, false);
      constexpr uint32_t idPV = idesc_f16(128, DV, BF16, false, true);
      const uint64_t dQ0 = sdesc_sw128(smem_u32(sQ), 16, 1024);  // Q tile 0, K-major (A of S)
      auto kstep = [](int kk, int rows) -> uint32_t { return (kk / 4) * (rows * 128) + (kk % 4) * 32; };
      bool ok = mbar_wait_warp(&ctl.bar_q, 0, guard, 2);
      // S_w of key tile j into warpgroup w's S columns
      auto issue_s = [&](int w, int j) {
        const int st = j % C::KST;
        const uint64_t dK = sdesc_sw128(smem_u32(sK0 + st * C::K_BYTES), 16, 1024);
        const uint64_t dQ = desc_advance(dQ0, w * C::Q_BYTES);
#pragma unroll 4
        for (int kk = 0; kk < DQK / 16; ++kk)
          umma_ss(tmem + w * C::WG_COLS, desc_advance(dQ, kstep(kk, C::BQ)), desc_advance(dK, kstep(kk, C::BK)),
                  idS, kk > 0);
        umma_commit(&ctl.s_full[w]);
      };
      // the two ranges packed as 16-bit halves, for the MMA warp's 24 registers (n <= 65535 128-key tiles:
      // the parameter check rejects longer sequences)
      const uint32_t r0 = static_cast<uint32_t>(jlo0) | (static_cast<uint32_t>(jhi0) << 16);
      const uint32_t r1 = static_cast<uint32_t>(jlo1) | (static_cast<uint32_t>(jhi1) << 16);
      // O_w += P_w . V of key tile j (A = P_w in TMEM, B = V read MN-major); the warpgroup's first tile
      // overwrites O
      auto first = [&](int w) -> int {
        if constexpr (C::OWN_RANGES) return static_cast<int>((w ? r1 : r0) & 0xffffu);
        else return 0;
      };
      auto issue_pv = [&](int w, int j) {
        const int vs = j % C::VST;
        const uint64_t dVmn = sdesc_sw128(smem_u32(sV0 + vs * C::V_BYTES), C::BK * 128, 1024);
        const uint32_t tO = tmem + w * C::WG_COLS + C::BK;
        const uint32_t tP = C::SEP_P ? tmem + C::P_COL + w * (C::BK / 2) : tmem + w * C::WG_COLS;
#pragma unroll
        for (int kk = 0; kk < C::BK / 16; ++kk)
          umma_ts(tO, tP + kk * 8, desc_advance(dVmn, kk * 2048), idPV, (j > first(w) || kk > 0) ? 1u : 0u);
      };
      auto mine = [&](int w, int j) -> bool {
        if constexpr (C::OWN_RANGES) {
          const uint32_t r = w ? r1 : r0;
          return j >= static_cast<int>(r & 0xffffu) && j < static_cast<int>(r >> 16);
        } else {
          return true;
        }
      };
      auto phase = [&](int w, int j) -> uint32_t { return static_cast<uint32_t>(j - first(w)) & 1u; };
      if (ok && n > 0) {
        ok = mbar_wait_warp(&ctl.k_full[0], 0, guard, 3);
        if (ok) {
          tc_fence_after();
          if constexpr (C::OWN_RANGES) {
            for (int w = 0; w < 2; ++w)
              if (mine(w, 0)) issue_s(w, 0);
          } else {
            issue_s(0, 0);
            issue_s(1, 0);
          }
          umma_commit(&ctl.k_empty[0]);
        }
      }
      // every barrier of warpgroup w completes one phase per tile of its own: phase(w, j)
      if constexpr (C::SEP_P) {
        // per key tile j, in the order the two warpgroups (half a tile apart) get there: S_0 of j + 1
        // once warpgroup 0 has read S_0 of j; P_1 . V of j - 1; S_1 of j + 1; P_0 . V of j
        for (int j = 0; ok && j < n; ++j) {
          const bool next = j + 1 < n;
          const int kn = (j + 1) % C::KST;
          if (next) {
            if (!mbar_wait_warp(&ctl.k_full[kn], ((j + 1) / C::KST) & 1, guard, 3)) { ok = false; break; }
            for (int w = 0; w < 2; ++w) {
              if (!mine(w, j + 1)) continue;
              if (mine(w, j)) {  // S_w of tile j read before the next S_w overwrites it
                if (!mbar_wait_warp(&ctl.s_free[w], phase(w, j), guard, 9)) { ok = false; break; }
                tc_fence_after();
              }
              issue_s(w, j + 1);
            }
            if (!ok) break;
            umma_commit(&ctl.k_empty[kn]);
          }
          if (!mbar_wait_warp(&ctl.v_full[j % C::VST], (j / C::VST) & 1, guard, 8)) { ok = false; break; }
          for (int w = 0; w < 2; ++w) {
            if (!mine(w, j)) continue;
            if (!mbar_wait_warp(&ctl.p_full[w], phase(w, j), guard, 5)) { ok = false; break; }
            tc_fence_after();
            issue_pv(w, j);
            umma_commit(&ctl.pv_done[w]);
          }
          if (!ok) break;
          umma_commit(&ctl.v_empty[j % C::VST]);
        }
      } else if constexpr (!C::OWN_RANGES) {
        // both warpgroups on every key tile of the union
        for (int j = 0; ok && j < n; ++j) {
          const bool next = j + 1 < n;
          const int kn = (j + 1) % C::KST;
          if (!mbar_wait_warp(&ctl.v_full[j % C::VST], (j / C::VST) & 1, guard, 8)) break;
          for (int w = 0; w < 2; ++w) {
            // P_w of tile j in TMEM over S_w: its P.V, then S_w of the next tile over the same columns
            // (tcgen05.mma runs in issue order, so P.V has read P before S overwrites it)
            if (!mbar_wait_warp(&ctl.p_full[w], j & 1, guard, 5)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv(w, j);
            if (next) {
              if (w == 0 && !mbar_wait_warp(&ctl.k_full[kn], ((j + 1) / C::KST) & 1, guard, 3)) {
                ok = false;
                break;
              }
              issue_s(w, j + 1);
            }
          }
          if (!ok) break;
          umma_commit(&ctl.v_empty[j % C::VST]);
          if (next) umma_commit(&ctl.k_empty[kn]);
        }
      } else {
        for (int j = 0; ok && j < n; ++j) {
          const bool next = j + 1 < n;
          const int kn = (j + 1) % C::KST;
          if (!mbar_wait_warp(&ctl.v_full[j % C::VST], (j / C::VST) & 1, guard, 8)) break;
          bool k_ready = false;
          for (int w = 0; w < 2; ++w) {
            // P_w of tile j in TMEM over S_w: its P.V, then S_w of the next tile over the same columns
            // (tcgen05.mma runs in issue order, so P.V has read P before S overwrites it)
            if (mine(w, j)) {
              if (!mbar_wait_warp(&ctl.p_full[w], phase(w, j), guard, 5)) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_pv(w, j);
            }
            if (next && mine(w, j + 1)) {
              if (!k_ready && !mbar_wait_warp(&ctl.k_full[kn], ((j + 1) / C::KST) & 1, guard, 3)) {
                ok = false;
                break;
              }
              k_ready = true;
              issue_s(w, j + 1);
            }
          }
          if (!ok) break;
          // a K stage no warpgroup reads has landed all the same before it is handed back
          if (next && !k_ready && !mbar_wait_warp(&ctl.k_full[kn], ((j + 1) / C::KST) & 1, guard, 3)) break;
          umma_commit(&ctl.v_empty[j % C::VST]);
          if (next) umma_commit(&ctl.k_empty[kn]);
        }
      }
      umma_commit(&ctl.acc_done);
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    reg_alloc<C::SOFTMAX_REGS>();
    const int w = warp >> 2;
    const int r = tid & 127;
    const int il = (2 * tp + w) * C::BQ + r;  // query row within the sequence
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + w * C::WG_COLS, tO = tS + C::BK;
    const uint32_t tP = C::SEP_P ? tmem + lane_base + C::P_COL + w * (C::BK / 2) : tS;
    const float sl2 = p.scale_log2;
    const float2 sl22 = make_float2(sl2, sl2);
    const float sink2 = sink ? __ldg(sink + h) * kLog2e : -INFINITY;
    // m_ref: the maximum P is taken against (-inf: nothing seen yet); l: row sum of P (the sink's term
    // e^{sink - m_ref} included)
    float mref = sink2;
    float l = sink ? 1.f : 0.f;
    bool ok = true;
    // this warpgroup's own key tiles: nw of them from key tile kw (local index jl)
    const int kw = k0 + (w ? jlo1 : jlo0), nw = w ? jhi1 - jlo1 : jhi0 - jlo0;
    for (int jl = 0; jl < nw; ++jl) {
      const int j0 = (kw + jl) * C::BK;
      const int i0 = (2 * tp + w) * C::BQ;
      // some key of the tile past the sequence's end, right of the first row's reach or left of the last
      // row's window
      const bool need_mask = (j0 + C::BK > sk.len) || (p.right > 0 && j0 + C::BK > i0 + off + p.right) ||
                             (p.window > 0 && i0 + C::BQ - 1 + off - j0 >= p.window);
      if (!mbar_wait_warp(&ctl.s_full[w], jl & 1, guard, 6)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // the whole S row into registers with one wait; S's columns are then free for the next tile's S
      uint32_t sv[C::BK];
      if constexpr (C::BK == 128) {
        tmem_ld128(tS, sv);
      } else {
        tmem_ld64(tS, sv);
      }
      if constexpr (C::SEP_P) {
        tc_fence_before();
        mbar_arrive_warp(&ctl.s_free[w]);
      }
      // one key tile of this warpgroup's rows, compiled with and without the mask (an unmasked tile then
      // works on S where the load put it)
      auto tile = [&](auto mask_tag) -> bool {
        constexpr bool MASK = decltype(mask_tag)::value;
        // the keys e of the tile this row sees form one interval lo <= e < hi: the key exists, lies left of
        // the row's reach (d > -right) and inside its window (d < window), d = i + off - key
        int lo = 0, hi = C::BK;
        if constexpr (MASK) {
          const long long d0 = static_cast<long long>(il) + off - j0;  // diagonal distance to the tile's first key
          long long h2 = sk.len - j0;
          if (p.right > 0 && d0 + p.right < h2) h2 = d0 + p.right;
          const long long l2 = p.window > 0 ? d0 - p.window + 1 : 0;
          hi = static_cast<int>(h2 < 0 ? 0 : (h2 > C::BK ? C::BK : h2));
          lo = static_cast<int>(l2 < 0 ? 0 : (l2 > C::BK ? C::BK : l2));
        }
        // S of 32 columns from the row in registers, masked (-inf) outside [lo, hi)
        auto cols = [&](int c, float (&x)[32]) {
#pragma unroll
          for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(sv[32 * c + e]);
          if constexpr (MASK) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (32 * c + e < lo || 32 * c + e >= hi) x[e] = -INFINITY;
          }
        };
        // the tile's maximum of S * scale * log2(e) over the keys the row sees, in fp32
        auto tile_max = [&]() -> float {
          float c0 = -INFINITY, c1 = -INFINITY;
#pragma unroll
          for (int c = 0; c < C::BK / 32; ++c) {
            float x[32];
            cols(c, x);
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              c0 = fmaxf(c0, x[e]);
              c1 = fmaxf(c1, x[e + 1]);
            }
          }
          return fmaxf(c0, c1) * sl2;  // scale > 0 commutes with the maximum
        };
        // a row that has seen no key yet (and has no sink) takes this tile's maximum as m_ref
        if (__any_sync(0xffffffffu, mref == -INFINITY)) {
          const float mt = tile_max();
          if (mref == -INFINITY) mref = mt;
        }
        float2 lsum[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        uint32_t pk[C::BK / 2];
        // P = exp2(S * scale * log2(e) - mu) of one 32-column chunk, packed (16 words) and added into the
        // row sums
        auto chunk = [&](int c, float mu) {
          float v[32];
          cols(c, v);
          const float2 nm = make_float2(-mu, -mu);
          if constexpr (BF16) {
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const float2 x0 = fma2(make_float2(v[e], v[e + 1]), sl22, nm);
              const float2 x1 = fma2(make_float2(v[e + 2], v[e + 3]), sl22, nm);
              const float2 p01 = make_float2(ex2_approx(x0.x), ex2_approx(x0.y));
              const float2 p23 = make_float2(ex2_approx(x1.x), ex2_approx(x1.y));
              lsum[0] = add2(lsum[0], p01);
              lsum[1] = add2(lsum[1], p23);
              pk[16 * c + e / 2] = pack2<true>(p01.x, p01.y);
              pk[16 * c + e / 2 + 1] = pack2<true>(p23.x, p23.y);
            }
          } else {
            // the argument rounded to fp16 and exponentiated two at a time
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              const float2 x0 = fma2(make_float2(v[e], v[e + 1]), sl22, nm);
              const float2 x1 = fma2(make_float2(v[e + 2], v[e + 3]), sl22, nm);
              pk[16 * c + e / 2] = ex2_f16x2(pack2<false>(x0.x, x0.y));
              pk[16 * c + e / 2 + 1] = ex2_f16x2(pack2<false>(x1.x, x1.y));
            }
            // the chunk's 32 values of P added in fp16: four partial sums of four pairs each, then
            // combined, then into the fp32 row sum
            auto hp = [&](int e) { return u32_as_half2(pk[16 * c + e]); };
            const __half2 a = __hadd2(__hadd2(hp(0), hp(4)), __hadd2(hp(8), hp(12)));
            const __half2 b = __hadd2(__hadd2(hp(1), hp(5)), __hadd2(hp(9), hp(13)));
            const __half2 d = __hadd2(__hadd2(hp(2), hp(6)), __hadd2(hp(10), hp(14)));
            const __half2 q = __hadd2(__hadd2(hp(3), hp(7)), __hadd2(hp(11), hp(15)));
            lsum[c & 1] = add2(lsum[c & 1], __half22float2(__hadd2(__hadd2(a, b), __hadd2(d, q))));
          }
        };
        // P of the whole tile against mu; returns its row sum
        auto pass = [&](float mu) -> float {
          lsum[0] = lsum[1] = make_float2(0.f, 0.f);
#pragma unroll
          for (int c = 0; c < C::BK / 32; ++c) chunk(c, mu);
          return (lsum[0].x + lsum[0].y) + (lsum[1].x + lsum[1].y);
        };
        float t = pass((mref == -INFINITY) ? 0.f : mref);
        // separate P: P . V of the previous tile has finished reading P and adding into O
        if (C::SEP_P && jl > 0) {
          if (!mbar_wait_warp(&ctl.pv_done[w], (jl - 1) & 1, guard, 10)) return false;
          tc_fence_after();
        }
        // every P of the tile is at most its row sum: a sum within 2^TAU keeps P <= 2^TAU.  Above it (or
        // not finite: an fp16 argument or P past fp16's range) m_ref moves to the tile's maximum -- the whole
        // warp, as TMEM loads and stores are warp-collective -- the O rows and the row sum are rescaled and
        // the tile's P computed again (then P <= 1)
        const bool need = !(t <= C::P_MAX);
        if (__any_sync(0xffffffffu, need)) {
          const float mnew = fmaxf(mref, tile_max());
          const float f = (mref == -INFINITY) ? 0.f : ex2_approx(mref - mnew);  // nothing accumulated yet: 0
          l *= f;
          if (jl > 0) {
#pragma unroll 1
            for (int c0 = 0; c0 < DV; c0 += 16) {
              uint32_t o[16];
              tmem_ld16(tO + c0, o);
#pragma unroll
              for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
              tmem_st16(tO + c0, o);
            }
          }
          mref = mnew;
          t = pass((mref == -INFINITY) ? 0.f : mref);
        }
#pragma unroll
        for (int c = 0; c < C::BK / 32; ++c) tmem_st16(tP + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(pk + 16 * c));
        l += t;
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive_warp(&ctl.p_full[w]);
        return true;
      };
      if (!(need_mask ? tile(std::true_type{}) : tile(std::false_type{}))) {
        ok = false;
        break;
      }
    }
    // epilogue: O = O_w / l, LSE = ln 2 * (m_ref + log2 l)
    if (ok && mbar_wait_warp(&ctl.acc_done, 0, guard, 7)) {
      tc_fence_after();
      const bool valid = il < sq.len;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      T* o = static_cast<T*>(out) + p.o_st.row(sq.b, h, sq.start + il);
#pragma unroll 1
      for (int c0 = 0; c0 < DV; c0 += 32) {
        uint32_t v[32];
        if (nw > 0) tmem_ld32(tO + c0, v);  // all lanes: .sync.aligned
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
      if (valid) {
        const float mu = (mref == -INFINITY) ? 0.f : mref;
        lse_out[static_cast<size_t>(zq) * p.S + sq.start + il] = (l > 0.f) ? (mu + log2f(l)) * kLn2 : -INFINITY;
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
static cudaError_t launch_fwd_t(const Problem& p, const Maps& m, const float* sink, void* out, float* lse,
                                cudaStream_t st) {
  using C = FwdCfg<DQK, DV, BF16>;
  auto kern = fwd_kernel<DQK, DV, BF16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  const int npair = (p.max_len + 2 * C::BQ - 1) / (2 * C::BQ);
  if (npair == 0 || p.nseqs == 0) return cudaSuccess;
  dim3 grid(p.Hq, npair, p.nseqs);
  kern<<<grid, C::THREADS, C::SMEM, st>>>(p, m, sink, out, lse);
  return cudaGetLastError();
}

cudaError_t launch_fwd(const Problem& p, int dtype_bf16, const Maps& m, const float* sink, void* o, float* lse,
                       cudaStream_t st) {
#define GQA_F(DQK, DV)                                                               \
  if (p.Dqk == DQK && p.Dv == DV)                                                    \
    return dtype_bf16 ? launch_fwd_t<DQK, DV, true>(p, m, sink, o, lse, st)           \
                      : launch_fwd_t<DQK, DV, false>(p, m, sink, o, lse, st);
  GQA_F(64, 64)
  GQA_F(128, 128)
  GQA_F(192, 128)
#undef GQA_F
  return cudaErrorInvalidValue;
}

int fwd_kernel_bk(int Dqk) { return Dqk <= 128 ? 128 : 64; }

}  // namespace gqa
