// Split-KV verify attention on the 5th-generation tensor core, for query blocks dense enough to
// be a real contraction (nq * G > 32 rows per kv head: the 70B-shaped chain with 7 x 8 = 56 rows,
// Medusa-style trees with 64 x 4 = 256 rows).
//
// Same stream-K decomposition, workspace records and merge kernel as the mma.sync path (attn.cu);
// one CTA per SM.  Per CTA, one 128-row block of query rows (a "row group"), warp-specialised:
//   warp 0     TMA producer: 128-key K and V tiles (128-byte swizzle) into a 3-stage ring.
//   warp 1     MMA issuer (one lane) and TMEM owner.
//   warps 2-9  two softmax warpgroups.  Warpgroup w takes the tiles of the CTA's walk whose
//              global index t has t mod 2 = w, with its own score buffer S_w and output
//              accumulator O_w in TMEM, so the two run their softmax concurrently (two warps per
//              SM sub-partition hide each other's latency) while the tensor core works for the
//              other one.
// Per tile t of warpgroup w: S_w = Q K_t^T (M = 128 rows, N = 128 keys, K = 128); the warpgroup
// reads S_w twice from TMEM, first for the row max, then for P = 2^(s * scale - mu) written as
// bf16 pairs over S_w's first 64 columns (each chunk's P lands on columns already read); then
// O_w += P V_t (P from TMEM, V as an MN-major shared-memory operand).  mu is a lazily updated row
// max: it moves (and O_w is rescaled in TMEM) only when a tile's max exceeds it by more than 2^8.
// The MMA issuer orders PV(t) before QK(t + 2) (same S_w), and the tcgen05.mma operations of one
// thread execute in issue order, so S_w is overwritten only after P_w has been consumed.
// At the end of each part each warpgroup writes its own (m, l, o) record: two key slices per part
// for the merge kernel.
// Query rows are spread over the four TMEM sub-partitions (row r -> lane 32 (r mod 4) + r / 4)
// so that a 56-row block keeps all four warps of a warpgroup busy.
// TMEM columns (512 allocated): S_0 [0,128), S_1 [128,256), O_0 [256,384), O_1 [384,512).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "attn_common.cuh"
#include "attn_internal.h"
#include "common.cuh"
#include "tcgen05.cuh"
#include "launch_cache.h"

namespace specv {

constexpr int kTcRows = 128;     // M: query rows per CTA
constexpr int kTcKeys = 128;     // keys per tile (N of QK^T, K of PV)
constexpr int kTcStages = 3;
constexpr int kTcD = 128;
constexpr uint32_t kTmemCols = 512;
constexpr int kTcThreads = 64 + kTcSlices * 128;   // TMA warp, MMA warp, softmax warpgroups
constexpr int kTile = kTcKeys * kTcD * 2;   // bytes of one K (or V) tile: 32 KB
constexpr int kHalf = kTcKeys * 128;        // one 64-column (128-byte) half of a tile: 16 KB
constexpr int kQHalf = kTcRows * 128;       // one half of the Q block: 16 KB
constexpr float kRescaleLog2 = 8.0f;        // lazy-rescale threshold: 2^8
constexpr uint32_t kColO = 2 * kTcKeys;     // TMEM column of O_0 (O_1 at +128)

constexpr uint32_t kIdescQK = tc::idesc_bf16(kTcRows, kTcKeys, 0, 0);  // A = Q (K-major), B = K (K-major)
constexpr uint32_t kIdescPV = tc::idesc_bf16(kTcRows, kTcD, 0, 1);     // A = P (TMEM), B = V (MN-major)

size_t attn_tc_smem_bytes() { return 1024 + (size_t)kTcStages * 2 * kTile + 2 * (size_t)kQHalf; }

__device__ __forceinline__ int tc_row_of_lane(int m) { return 4 * (m & 31) + (m >> 5); }

// The global tile sequence of a CTA's walk: tile t is tile i of the n tiles of part `part`.
struct TcTile {
  int valid, part, i, n;
};

struct TcIter {
  Walker w;
  int part, i, n;
};

__device__ __forceinline__ void tc_iter_init(const AttnParams& p, int cta, TcIter& it) {
  walker_init(p, cta, it.w);
  it.part = -1;
  it.i = 0;
  it.n = 0;
}

__device__ __forceinline__ TcTile tc_iter_next(const AttnParams& p, TcIter& it) {
  TcTile t{0, 0, 0, 0};
  if (it.i == it.n) {
    int b, g, kb, ke, len;
    if (!walker_next(p, it.w, b, g, kb, ke, len)) return t;
    ++it.part;
    it.i = 0;
    it.n = (ke - kb + kTcKeys - 1) / kTcKeys;
  }
  t.valid = 1;
  t.part = it.part;
  t.i = it.i++;
  t.n = it.n;
  return t;
}

template <int MASK>
__global__ void __launch_bounds__(kTcThreads, 1)
    attn_partial_tc(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ AttnParams p) {
  pdl_launch_dependents();  // the merge may be scheduled as SMs free up
  // the call's status word is cleared here (no memset node before the call's first kernel)
  if (blockIdx.x == 0 && threadIdx.x == 0) status_clear_for_launch(p.status);
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[kTcStages], empty[kTcStages];
  __shared__ uint64_t sfull[kTcSlices], pfull[kTcSlices], pvdone[kTcSlices], ofree[kTcSlices];
  __shared__ uint64_t qfull, drain;
  __shared__ uint32_t tmem_base;
  __shared__ int s_abort;

  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* stages = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* sQ = stages + kTcStages * 2 * kTile;
  const uint32_t stages_u32 = smem_u32(stages), sQ_u32 = smem_u32(sQ);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int groups = p.tc_groups;
  const int cta = blockIdx.x / groups;                 // key range
  const int row0 = (blockIdx.x % groups) * p.rows_per_group;
  const int rows_here = min(p.rows_per_group, p.rows - row0);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kTcStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < kTcSlices; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&pfull[i], 4);
      mbar_init(&pvdone[i], 1);
      mbar_init(&ofree[i], 4);
    }
    mbar_init(&qfull, 4);
    mbar_init(&drain, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tc::alloc(&tmem_base, kTmemCols);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_base;

  auto fail = [&]() {
    s_abort = 1;
    status_report(p.status, (uint32_t)SPEC_STATUS_TIMEOUT);
  };

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    Walker w;
    walker_init(p, cta, w);
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int t = 0;
      bool ok = true;
      int b, g, kb, ke, len;
      while (ok && !p.debug_no_loads && walker_next(p, w, b, g, kb, ke, len)) {
        for (int key0 = kb; key0 < ke; key0 += kTcKeys, ++t) {
          const int s = t % kTcStages;
          if (!mbar_wait_bounded(&empty[s], ((t / kTcStages) & 1) ^ 1u, &s_abort)) {
            fail();
            ok = false;
            break;
          }
          uint8_t* sk = stages + s * 2 * kTile;
          mbar_arrive_expect_tx(&full[s], 2u * kTile);
          tma_load_kv(sk, &tmK, &full[s], key0, g, b);
          tma_load_kv(sk + kTile, &tmV, &full[s], key0, g, b);
        }
      }
      if (!ok || s_abort) {
        for (int i = 1; i <= min(t, kTcStages); ++i) {  // copies still in flight into this CTA
          const int tt = t - i;
          mbar_wait_bounded(&full[tt % kTcStages], (tt / kTcStages) & 1, nullptr);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // Issue order: QK(0), QK(1), then for t = 0, 1, ...: PV(t), QK(t + 2).
    TcIter it;
    tc_iter_init(p, cta, it);
    if (lane == 0) {
      bool ok = true;
      auto issue_qk = [&](int t, const TcTile& T) -> bool {
        if (T.i == 0 && !mbar_wait_bounded(&qfull, T.part & 1, &s_abort)) return false;
        const int s = t % kTcStages;
        if (!mbar_wait_bounded(&full[s], (t / kTcStages) & 1, &s_abort)) return false;
        tc::fence_after();
        const uint32_t kbase = stages_u32 + s * 2 * kTile;
        const uint32_t d = tmem + (uint32_t)(t & 1) * kTcKeys;
#pragma unroll
        for (int ks = 0; ks < kTcD / 16; ++ks) {
          const uint64_t adesc = tc::smem_desc(sQ_u32 + (ks >> 2) * kQHalf + (ks & 3) * 32, 16, 1024);
          const uint64_t bdesc = tc::smem_desc(kbase + (ks >> 2) * kHalf + (ks & 3) * 32, 16, 1024);
          tc::mma_ss(d, adesc, bdesc, kIdescQK, ks > 0 ? 1u : 0u);
        }
        tc::commit(&sfull[t & 1]);
        return true;
      };
      auto issue_pv = [&](int t, const TcTile& T) -> bool {
        const int wg = t & 1;
        const bool wg_first = T.i < 2;  // the warpgroup's first tile of the part
        if (wg_first && T.part >= 1 && !mbar_wait_bounded(&ofree[wg], (T.part - 1) & 1, &s_abort)) return false;
        if (!mbar_wait_bounded(&pfull[wg], (t >> 1) & 1, &s_abort)) return false;
        tc::fence_after();
        const uint32_t vb = stages_u32 + (t % kTcStages) * 2 * kTile + kTile;
        const uint32_t pa = tmem + (uint32_t)wg * kTcKeys;
        const uint32_t od = tmem + kColO + (uint32_t)wg * kTcD;
#pragma unroll
        for (int ks = 0; ks < kTcKeys / 16; ++ks) {
          const uint64_t bdesc = tc::smem_desc(vb + ks * 2048, kHalf, 1024);
          tc::mma_ts(od, pa + ks * 8, bdesc, kIdescPV, (ks > 0 || !wg_first) ? 1u : 0u);
        }
        tc::commit(&pvdone[wg]);
        tc::commit(&empty[t % kTcStages]);
        return true;
      };
      const TcTile none{0, 0, 0, 0};
      TcTile ring[3];
      ring[0] = tc_iter_next(p, it);
      ring[1] = ring[0].valid ? tc_iter_next(p, it) : none;
      if (ring[0].valid && !issue_qk(0, ring[0])) ok = false;
      if (ok && ring[1].valid && !issue_qk(1, ring[1])) ok = false;
      for (int t = 0; ok && ring[t % 3].valid; ++t) {
        ring[(t + 2) % 3] = ring[(t + 1) % 3].valid ? tc_iter_next(p, it) : none;
        if (!issue_pv(t, ring[t % 3])) { ok = false; break; }
        if (ring[(t + 2) % 3].valid && !issue_qk(t + 2, ring[(t + 2) % 3])) { ok = false; break; }
      }
      if (!ok) {
        fail();
        tc::commit(&drain);  // every MMA issued so far has finished before TMEM is released
        mbar_wait_bounded(&drain, 0, nullptr);
      }
    }
  } else {
    // ------------------------------------------------------------------ softmax warpgroups
    const int wg = (warp - 2) >> 2;                // this warpgroup takes the tiles with t mod 2 = wg
    const int sub = warp & 3;                      // TMEM sub-partition of this warp
    const int m = sub * 32 + lane;                 // TMEM lane = M row
    const int r = tc_row_of_lane(m);               // query row within the row group
    const bool real = r < rows_here;
    const int rr = row0 + r;
    const int jq = real ? rr / p.G : 0;            // query position (chain row / tree node)
    const unsigned long long anc = (MASK == kMaskTree && real) ? p.anc[jq] : 0ull;
    const uint32_t tl = tmem + ((uint32_t)(sub * 32) << 16);
    const uint32_t sbuf = tl + (uint32_t)wg * kTcKeys;         // S_w (P_w over its first 64 columns)
    const uint32_t obuf = tl + kColO + (uint32_t)wg * kTcD;    // O_w
    const __nv_bfloat16* qbase = reinterpret_cast<const __nv_bfloat16*>(p.q);
    const int stid = (threadIdx.x - 64) & 127;     // 0..127 within the warpgroup
    const float sc = p.scale_log2;

    // Q block of (b, g) into shared memory (K-major, 128-byte swizzle); one arrival per warp.
    auto load_q = [&](int b, int g) {
      uint4 v[16];
      if (real) {
        const uint4* src = reinterpret_cast<const uint4*>(qbase + b * p.q_sb + (int64_t)jq * p.q_st +
                                                          (int64_t)(g * p.G + rr % p.G) * p.q_sh);
#pragma unroll
        for (int c = 0; c < 16; ++c) v[c] = src[c];
      } else {
#pragma unroll
        for (int c = 0; c < 16; ++c) v[c] = make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int cc = c & 7;
        *reinterpret_cast<uint4*>(sQ + (c >> 3) * kQHalf + (m >> 3) * 1024 + (m & 7) * 128 + ((cc ^ (m & 7)) << 4)) =
            v[c];
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&qfull);
    };

    // all lanes wait, then re-converge (the TMEM accesses that follow are warp-collective)
    auto warp_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
      const bool got = mbar_wait_bounded(bar, parity, &s_abort);
      return __all_sync(0xffffffffu, got);
    };

    Walker w;
    walker_init(p, cta, w);
    int b, g, kb, ke, len;
    bool have = walker_next(p, w, b, g, kb, ke, len);
    if (have && wg == 0) load_q(b, g);  // the first part's Q; later ones follow a part's last tile
    int t0 = 0;       // global index of the part's first tile
    int kt = 0;       // this warpgroup's tiles so far (phase counter of sfull / pfull / pvdone)
    int pv_seen = 0;  // pvdone phases of this warpgroup observed so far
    bool ok = true;
    while (have && ok) {
      const int n = (ke - kb + kTcKeys - 1) / kTcKeys;
      int nb = 0, ng = 0, nkb = 0, nke = 0, nlen = 0;
      const bool have_next = walker_next(p, w, nb, ng, nkb, nke, nlen);
      const int tail_start = len - p.nq;
      float m_run = neg_inf(), l = 0.f;
      int mine = 0;
      for (int i = ((t0 & 1) == wg) ? 0 : 1; i < n; i += 2) {
        const int t = t0 + i;
        const int key0 = kb + i * kTcKeys;
        if (!warp_wait(&sfull[wg], kt & 1)) { ok = false; break; }
        tc::fence_after();
        // the part's last scores are in, so every Q K^T of the part has completed: next Q
        if (i == n - 1 && have_next) load_q(nb, ng);
        const bool edge = key0 + kTcKeys > ke || (MASK != kMaskNone && key0 + kTcKeys > tail_start);
        // V rows of keys at or past the sequence end may hold anything (NaN): zero them before P.V
        if (key0 + kTcKeys > len) {
          const int s = t % kTcStages;
          if (!warp_wait(&full[s], (t / kTcStages) & 1)) { ok = false; break; }
          uint8_t* vb = stages + s * 2 * kTile + kTile;
          const int vrow0 = max(len - key0, 0);
          for (int idx = stid; idx < (kTcKeys - vrow0) * 16; idx += 128) {
            const int row = vrow0 + idx / 16, c = idx % 16;
            *reinterpret_cast<uint4*>(vb + (c >> 3) * kHalf + row * 128 + (c & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          tc::fence_proxy_async_smem();
          __syncwarp();
        }
        // ---- pass 1: the row's largest visible scaled score in this tile
        float tmax;
        {
          float mx[4] = {neg_inf(), neg_inf(), neg_inf(), neg_inf()};
          uint32_t u[32];
#pragma unroll 1
          for (int c4 = 0; c4 < 4; ++c4) {
            tc::ld32(sbuf + c4 * 32, u);
            tc::ld_wait(u);
            if (!edge) {
#pragma unroll
              for (int e = 0; e < 32; ++e) mx[e & 3] = fmaxf(mx[e & 3], __uint_as_float(u[e]));
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                const bool vis = key_visible_nb<MASK>(key0 + c4 * 32 + e, ke, tail_start, jq, anc);
                mx[e & 3] = fmaxf(mx[e & 3], vis ? __uint_as_float(u[e]) : neg_inf());
              }
            }
          }
          const float raw_max = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
          tmax = (real && raw_max != neg_inf()) ? raw_max * sc : neg_inf();
        }
        // ---- reference max: the first tile of the part sets it; afterwards it moves (and O_w
        // is rescaled) only when the tile max exceeds it by more than 2^8
        if (mine == 0) {
          m_run = tmax;
        } else {
          const bool need = tmax > m_run + kRescaleLog2 || (m_run == neg_inf() && tmax > neg_inf());
          if (__any_sync(0xffffffffu, need)) {
            // O_w may only be touched once this warpgroup's previous P.V has completed
            if (pv_seen < kt) {
              if (!warp_wait(&pvdone[wg], (kt - 1) & 1)) { ok = false; break; }
              pv_seen = kt;
              tc::fence_after();
            }
            float alpha = 1.f;
            if (need) {
              alpha = m_run == neg_inf() ? 0.f : ex2_approx(m_run - tmax);
              l *= alpha;
              m_run = tmax;
            }
            uint32_t u[32];
#pragma unroll 1
            for (int c4 = 0; c4 < 4; ++c4) {
              tc::ld32(obuf + c4 * 32, u);
              tc::ld_wait(u);
#pragma unroll
              for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
              tc::st32(obuf + c4 * 32, u);
            }
            tc::st_wait();
          }
        }
        ++mine;
        // ---- pass 2: P = 2^(s * scale - mu) as bf16 pairs over S_w's first 64 columns; the next
        // chunk's load is in flight while the current one is computed
        {
          const float mu = m_run == neg_inf() ? 0.f : m_run;
          float sums[4] = {0.f, 0.f, 0.f, 0.f};
          auto chunk = [&](const uint32_t (&u)[32], int c4) {
            uint32_t pk[16];
            if (!edge) {
#pragma unroll
              for (int e = 0; e < 32; e += 2) {
                const float p0 = ex2_approx(fmaf(__uint_as_float(u[e]), sc, -mu));
                const float p1 = ex2_approx(fmaf(__uint_as_float(u[e + 1]), sc, -mu));
                sums[(e >> 1) & 3] += p0 + p1;
                pk[e / 2] = pack_bf16(p0, p1);
              }
            } else {
#pragma unroll
              for (int e = 0; e < 32; e += 2) {
                const int kk = key0 + c4 * 32 + e;
                float x0 = fmaf(__uint_as_float(u[e]), sc, -mu);
                float x1 = fmaf(__uint_as_float(u[e + 1]), sc, -mu);
                x0 = (real & key_visible_nb<MASK>(kk, ke, tail_start, jq, anc)) ? x0 : neg_inf();
                x1 = (real & key_visible_nb<MASK>(kk + 1, ke, tail_start, jq, anc)) ? x1 : neg_inf();
                const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                sums[(e >> 1) & 3] += p0 + p1;
                pk[e / 2] = pack_bf16(p0, p1);
              }
            }
            __syncwarp();
            tc::st16(sbuf + c4 * 16, pk);
          };
          uint32_t ua[32], ub[32];
          tc::ld32(sbuf, ua);
          tc::ld_wait(ua);
          tc::ld32(sbuf + 32, ub);
          chunk(ua, 0);
          tc::ld_wait(ub);
          tc::ld32(sbuf + 64, ua);
          chunk(ub, 1);
          tc::ld_wait(ua);
          tc::ld32(sbuf + 96, ub);
          chunk(ua, 2);
          tc::ld_wait(ub);
          chunk(ub, 3);
          tc::st_wait();
          l += real ? (sums[0] + sums[1]) + (sums[2] + sums[3]) : 0.f;
        }
        // observe the warpgroup's previous P.V completion before this tile's P is handed over,
        // so that its P.V barrier never runs two phases ahead
        if (pv_seen < kt) {
          if (!warp_wait(&pvdone[wg], (kt - 1) & 1)) { ok = false; break; }
          pv_seen = kt;
        }
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pfull[wg]);
        ++kt;
      }
      if (!ok) break;
      // ---- epilogue: this warpgroup's (m, l, o) record of the part
      {
        const int64_t slot = (int64_t)(b * p.Hkv + g) + cta;
        const int64_t rec = (slot * kTcSlices + wg) * p.rows + rr;
        if (mine > 0) {
          if (pv_seen < kt) {
            if (!warp_wait(&pvdone[wg], (kt - 1) & 1)) { ok = false; break; }
            pv_seen = kt;
          }
          __syncwarp();
          tc::fence_after();
          uint32_t u[32];
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            __syncwarp();
            tc::ld32(obuf + c4 * 32, u);
            tc::ld_wait(u);
            if (real) {
              float4* dst = reinterpret_cast<float4*>(p.part_o + rec * kTcD + c4 * 32);
#pragma unroll
              for (int e = 0; e < 8; ++e)
                dst[e] = make_float4(__uint_as_float(u[4 * e]), __uint_as_float(u[4 * e + 1]),
                                     __uint_as_float(u[4 * e + 2]), __uint_as_float(u[4 * e + 3]));
            }
          }
          if (real) p.part_ml[rec] = make_float2(m_run, l);
        } else if (real) {
          // a one-tile part that went to the other warpgroup: an empty record
          float4* dst = reinterpret_cast<float4*>(p.part_o + rec * kTcD);
#pragma unroll 4
          for (int e = 0; e < kTcD / 4; ++e) dst[e] = make_float4(0.f, 0.f, 0.f, 0.f);
          p.part_ml[rec] = make_float2(neg_inf(), 0.f);
        }
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ofree[wg]);
      t0 += n;
      have = have_next;
      b = nb; g = ng; kb = nkb; ke = nke; len = nlen;
    }
    if (!ok) fail();
  }

  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc::fence_after();
    tc::dealloc(tmem, kTmemCols);
  }
}

template <int MASK>
static cudaError_t launch_tc_mask(const AttnParams& p, const CUtensorMap* tmK, const CUtensorMap* tmV,
                                  cudaStream_t stream) {
  const size_t smem = attn_tc_smem_bytes();
  auto kern = attn_partial_tc<MASK>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<p.grid_x * p.tc_groups, kTcThreads, smem, stream>>>(*tmK, *tmV, p);
  return cudaGetLastError();
}

cudaError_t launch_partial_tc(const AttnParams& p, const CUtensorMap* tmK, const CUtensorMap* tmV,
                              cudaStream_t stream) {
  if (p.nks != kTcSlices) return cudaErrorInvalidValue;
  switch (p.mask) {
    case kMaskNone: return launch_tc_mask<kMaskNone>(p, tmK, tmV, stream);
    case kMaskChain: return launch_tc_mask<kMaskChain>(p, tmK, tmV, stream);
    default: return launch_tc_mask<kMaskTree>(p, tmK, tmV, stream);
  }
}

}  // namespace specv
