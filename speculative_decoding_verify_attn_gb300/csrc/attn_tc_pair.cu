// Split-KV verify attention on the 5th-generation tensor core for more than 128 query rows per kv
// head (Medusa-style trees: 64 nodes x 4 heads = 256 rows): one CTA holds a pair of 128-row blocks
// and every K/V tile it loads serves both, so each tile crosses from L2 to the SM once for up to
// 256 rows.
//
// Same stream-K decomposition, workspace records (one per row and part) and merge kernel as the
// other attention kernels; one CTA per SM, warp-specialised:
//   warp 0       TMA producer: 64-key K and V tiles (128-byte swizzle) into a 5-stage ring.
//   warps 1, 2   MMA issuers (one lane each), warp 1 for row block 0, warp 2 for row block 1.
//                Two issuers keep the tensor pipe fed: its issue queue is shallow, and every
//                barrier wait of an issuing thread otherwise leaves the pipe idle.
//   warps 3-10   two softmax warpgroups; warpgroup w owns row block w of the pair.
// Per tile t and block w: S_w(t) = Q_w K_t^T (M = 128, N = 64, K = 128; Q_w and K_t in shared
// memory) into TMEM buffer t & 1; the warpgroup reads S_w(t) once, writes P = 2^(s * scale - mu)
// as bf16 pairs over the buffer's first 32 columns; O_w += P_w(t) V_t (P from TMEM, V as an
// MN-major shared-memory operand).  With two S buffers, issuer w puts Q K^T of tile t + 2 behind
// P.V of tile t, so the warpgroup's next scores are ready when it finishes a tile.  mu is the
// lazily updated row max of the other tensor-core kernel (O_w rescaled in TMEM only when a tile's
// max exceeds it by more than 2^8).  A stage is free once both issuers' P.V of its tile completed
// (two commits on its `empty` barrier).  P.V completions are signalled per S buffer (pvdone[w][t & 1]:
// phase t >> 1 of that barrier is P.V(t)), so a warpgroup waits for one only where it touches O (a
// rescale, the part's epilogue) and never needs to observe each of them to keep count.
// TMEM columns (512): block w at 256 w: S buffers [0,64) and [64,128), O [128,256).
// Query row m of a block is TMEM lane m and row m of the Q tile.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "attn_common.cuh"
#include "attn_internal.h"
#include "common.cuh"
#include "tcgen05.cuh"
#include "launch_cache.h"

namespace specv {

constexpr int kPRows = 128;                 // M: query rows per warpgroup
constexpr int kPKeys = kPairTileKeys;       // keys per tile (N of QK^T, K of PV)
constexpr int kPStages = 5;
constexpr int kPD = 128;
constexpr uint32_t kPTmemCols = 512;
constexpr int kPThreads = 96 + 2 * 128;     // TMA warp, two MMA warps, two softmax warpgroups
constexpr int kPTile = kPKeys * kPD * 2;    // bytes of one K (or V) tile: 16 KB
constexpr int kPHalf = kPKeys * 128;        // one 64-column (128-byte) half of a K/V tile: 8 KB
constexpr int kPQHalf = kPRows * 128;       // one 64-column half of a Q block: 16 KB
constexpr int kPQBlock = 2 * kPQHalf;       // one Q block: 32 KB
constexpr float kPRescaleLog2 = 8.0f;

__device__ __forceinline__ uint32_t p_col_s(int w, int buf) { return (uint32_t)(256 * w + kPKeys * buf); }
__device__ __forceinline__ uint32_t p_col_o(int w) { return (uint32_t)(256 * w + 2 * kPKeys); }

constexpr uint32_t kPIdescQK = tc::idesc_bf16(kPRows, kPKeys, 0, 0);  // A = Q, B = K (both K-major)
constexpr uint32_t kPIdescPV = tc::idesc_bf16(kPRows, kPD, 0, 1);     // A = P (TMEM), B = V (MN-major)

size_t attn_tc_pair_smem_bytes() { return 1024 + 2 * (size_t)kPQBlock + (size_t)kPStages * 2 * kPTile; }

// Sub-tiles of kPKeys keys over a CTA's walk: tile i of the n tiles of part `part`.
struct PTile {
  int valid, part, i, n;
};
struct PIter {
  Walker w;
  int part, i, n;
};
__device__ __forceinline__ void p_iter_init(const AttnParams& p, int cta, PIter& it) {
  walker_init(p, cta, it.w);
  it.part = -1;
  it.i = 0;
  it.n = 0;
}
__device__ __forceinline__ PTile p_iter_next(const AttnParams& p, PIter& it) {
  PTile t{0, 0, 0, 0};
  if (it.i == it.n) {
    int b, g, kb, ke, len;
    if (!walker_next(p, it.w, b, g, kb, ke, len)) return t;
    ++it.part;
    it.i = 0;
    it.n = (ke - kb + kPKeys - 1) / kPKeys;
  }
  t.valid = 1;
  t.part = it.part;
  t.i = it.i++;
  t.n = it.n;
  return t;
}

// Query row rr of (b, g) as row m of a Q block in shared memory, K-major with the 128-byte
// swizzle (16-byte chunk c of a 128-byte row stored at chunk c ^ (m & 7)); zeros for padding rows.
__device__ __forceinline__ void p_store_q(const AttnParams& p, bool real, int jq, int rr, int b, int g,
                                          uint8_t* qblock, int m) {
  const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.q) + b * p.q_sb +
                                                    (int64_t)jq * p.q_st + (int64_t)(g * p.G + rr % p.G) * p.q_sh);
  uint4 v[16];
#pragma unroll
  for (int c = 0; c < 16; ++c) v[c] = real ? src[c] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
  for (int c = 0; c < 16; ++c)
    *reinterpret_cast<uint4*>(qblock + (c >> 3) * kPQHalf + m * 128 + (((c & 7) ^ (m & 7)) << 4)) = v[c];
}

// Visibility of keys key0 .. key0 + 63 to query position jq as a bit mask (bit e: key key0 + e):
// keys before the part end ke; past tail_start (the verified positions) the chain rule (tail key
// m visible iff m <= jq) or the tree rule (iff bit m of the query's ancestor mask is set).
template <int MASK>
__device__ __forceinline__ unsigned long long p_tile_vis(int key0, int ke, int tail_start, int jq,
                                                         unsigned long long anc) {
  const int lim = ke - key0;
  const unsigned long long in = lim >= 64 ? ~0ull : (lim <= 0 ? 0ull : (1ull << lim) - 1ull);
  if (MASK == kMaskNone) return in;
  const int off = tail_start - key0;  // bit of the first tail key
  unsigned long long vis;
  if (off >= 64) {
    vis = ~0ull;
  } else if (MASK == kMaskChain) {
    const int last = off + jq;  // last visible bit
    vis = last >= 63 ? ~0ull : (last < 0 ? 0ull : (2ull << last) - 1ull);
  } else if (off > 0) {
    vis = ((1ull << off) - 1ull) | (anc << off);
  } else {
    vis = off > -64 ? anc >> (-off) : 0ull;
  }
  return in & vis;
}

// V rows of keys at or past the sequence end may hold anything (NaN): zero them before P.V
// (the 128 threads of one warpgroup; both warpgroups write the same zeros).
__device__ __forceinline__ void p_zero_v_tail(uint8_t* vb, int key0, int len, int stid) {
  const int vrow0 = max(len - key0, 0);
  for (int idx = stid; idx < (kPKeys - vrow0) * 16; idx += 128) {
    const int row = vrow0 + idx / 16, c = idx % 16;
    *reinterpret_cast<uint4*>(vb + (c >> 3) * kPHalf + row * 128 + (c & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
  }
}

template <int MASK>
__global__ void __launch_bounds__(kPThreads, 1)
    attn_partial_tc_pair(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ AttnParams p) {
  pdl_launch_dependents();  // the merge may be scheduled as SMs free up
  // the call's status word is cleared here (no memset node before the call's first kernel)
  if (blockIdx.x == 0 && threadIdx.x == 0) status_clear_for_launch(p.status);
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[kPStages], empty[kPStages];
  __shared__ uint64_t sfull[2][2], pfull[2][2], pvdone[2][2], ofree[2], qfull[2], drain[2];
  __shared__ uint64_t qfirst[2];  // q_tma: the first part's Q rows of each block, by TMA
  __shared__ uint32_t tmem_base;
  __shared__ int s_abort;

  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* qs = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // [block][half][128 rows][128 B]
  uint8_t* stages = qs + 2 * kPQBlock;                          // [stage][K tile, V tile]
  const uint32_t qs_u32 = smem_u32(qs);
  const uint32_t stages_u32 = smem_u32(stages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pairs = (p.tc_groups + 1) / 2;
  const int cta = blockIdx.x / pairs;  // key range
  const int pair = blockIdx.x % pairs;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kPStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 2);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(&sfull[w][0], 1);
      mbar_init(&sfull[w][1], 1);
      mbar_init(&pfull[w][0], 4);
      mbar_init(&pfull[w][1], 4);
      mbar_init(&pvdone[w][0], 1);
      mbar_init(&pvdone[w][1], 1);
      mbar_init(&ofree[w], 4);
      mbar_init(&qfull[w], 4);
      mbar_init(&qfirst[w], 1);
      mbar_init(&drain[w], 1);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) tc::alloc(&tmem_base, kPTmemCols);
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
      // q_tma: the first part's Q rows of both blocks are the CTA's first copies (the rows of a
      // block are 128 / G consecutive positions x the G heads of kv head g: one box per half of D)
      bool q_issued = false;
      if (p.q_tma && !p.debug_no_loads) {
        Walker w0 = w;
        int b0, g0, kb0, ke0, len0;
        if (walker_next(p, w0, b0, g0, kb0, ke0, len0)) {
          tma_prefetch_desc(&tmQ);
          for (int blk = 0; blk < 2; ++blk) {
            const int j0 = ((2 * pair + blk) * p.rows_per_group) / p.G;
            uint8_t* qb = qs + blk * kPQBlock;
            mbar_arrive_expect_tx(&qfirst[blk], (uint32_t)kPQBlock);
            tma_load_4d(qb, &tmQ, &qfirst[blk], 0, g0 * p.G, j0, b0);
            tma_load_4d(qb + kPQHalf, &tmQ, &qfirst[blk], 64, g0 * p.G, j0, b0);
          }
          q_issued = true;
        }
      }
      // every K/V tile is read once: let it leave L2 first (the records and Q stay)
      const uint64_t pol = l2_policy_evict_first();
      int t = 0;
      bool ok = true;
      int b, g, kb, ke, len;
      while (ok && !p.debug_no_loads && walker_next(p, w, b, g, kb, ke, len)) {
        for (int key0 = kb; key0 < ke; key0 += kPKeys, ++t) {
          const int s = t % kPStages;
          if (!mbar_wait_bounded(&empty[s], ((t / kPStages) & 1) ^ 1u, &s_abort)) {
            fail();
            ok = false;
            break;
          }
          uint8_t* sk = stages + s * 2 * kPTile;
          mbar_arrive_expect_tx(&full[s], 2u * kPTile);
          tma_load_kv_hint(sk, &tmK, &full[s], key0, g, b, pol);
          tma_load_kv_hint(sk + kPTile, &tmV, &full[s], key0, g, b, pol);
          // the first part's Q rows as plain loads by the softmax threads would queue behind
          // every CTA's ring fill (~25 MB of copies), so after the first tile the rest of the ring
          // waits until both row blocks' Q rows have landed
          if (t == 0 && !p.q_tma &&
              (!mbar_wait_bounded(&qfull[0], 0, &s_abort) || !mbar_wait_bounded(&qfull[1], 0, &s_abort))) {
            fail();
            ok = false;
            ++t;
            break;
          }
        }
      }
      if (!ok || s_abort) {
        for (int i = 1; i <= min(t, kPStages); ++i) {  // copies still in flight into this CTA
          const int tt = t - i;
          mbar_wait_bounded(&full[tt % kPStages], (tt / kPStages) & 1, nullptr);
        }
        if (q_issued) {
          mbar_wait_bounded(&qfirst[0], 0, nullptr);
          mbar_wait_bounded(&qfirst[1], 0, nullptr);
        }
      }
    }
  } else if (warp <= 2) {
    // ------------------------------------------------------------------ MMA issuer of block wm
    const int wm = warp - 1;
    PIter it;
    p_iter_init(p, cta, it);
    if (lane == 0) {
      const uint32_t qa0 = qs_u32 + wm * kPQBlock;
      // S_wm(t) = Q K_t^T into S buffer t & 1
      auto issue_qk = [&](int t, const PTile& T) -> bool {
        if (T.i == 0) {
          // the part's Q rows: by TMA for the first part (q_tma), else stored by the softmax warps
          const bool by_tma = p.q_tma && T.part == 0;
          if (!mbar_wait_bounded(by_tma ? &qfirst[wm] : &qfull[wm], by_tma ? 0u : (uint32_t)((T.part - p.q_tma) & 1),
                                 &s_abort))
            return false;
        }
        const int s = t % kPStages;
        if (!mbar_wait_bounded(&full[s], (t / kPStages) & 1, &s_abort)) return false;
        tc::fence_after();
        const uint32_t kbase = stages_u32 + s * 2 * kPTile;
        const uint32_t d = tmem + p_col_s(wm, t & 1);
#pragma unroll
        for (int ks = 0; ks < kPD / 16; ++ks) {
          const uint32_t koff = (ks >> 2) * kPHalf + (ks & 3) * 32;
          const uint64_t adesc = tc::smem_desc(qa0 + (ks >> 2) * kPQHalf + (ks & 3) * 32, 16, 1024);
          const uint64_t bdesc = tc::smem_desc(kbase + koff, 16, 1024);
          tc::mma_ss(d, adesc, bdesc, kPIdescQK, ks > 0 ? 1u : 0u);
        }
        tc::commit(&sfull[wm][t & 1]);
        return true;
      };
      // O_wm += P_wm(t) V_t; frees the stage once the other block's P.V of the tile is done too
      auto issue_pv = [&](int t, const PTile& T) -> bool {
        if (T.i == 0 && T.part >= 1 && !mbar_wait_bounded(&ofree[wm], (T.part - 1) & 1, &s_abort)) return false;
        if (!mbar_wait_bounded(&pfull[wm][t & 1], (t >> 1) & 1, &s_abort)) return false;
        tc::fence_after();
        const uint32_t vb = stages_u32 + (t % kPStages) * 2 * kPTile + kPTile;
        const uint32_t pa = tmem + p_col_s(wm, t & 1);
        const uint32_t od = tmem + p_col_o(wm);
#pragma unroll
        for (int ks = 0; ks < kPKeys / 16; ++ks) {
          const uint64_t bdesc = tc::smem_desc(vb + ks * 2048, kPHalf, 1024);
          tc::mma_ts(od, pa + ks * 8, bdesc, kPIdescPV, (ks > 0 || T.i > 0) ? 1u : 0u);
        }
        tc::commit(&pvdone[wm][t & 1]);
        tc::commit(&empty[t % kPStages]);
        return true;
      };
      bool ok = true;
      PTile cur = p_iter_next(p, it);
      PTile nxt = p_iter_next(p, it);
      if (cur.valid && !issue_qk(0, cur)) ok = false;
      if (ok && nxt.valid && !issue_qk(1, nxt)) ok = false;
      for (int t = 0; ok && cur.valid; ++t) {
        const PTile far = p_iter_next(p, it);  // tile t + 2
        if (!issue_pv(t, cur)) { ok = false; break; }
        if (far.valid && !issue_qk(t + 2, far)) { ok = false; break; }
        cur = nxt;
        nxt = far;
      }
      if (!ok) {
        fail();
        tc::commit(&drain[wm]);  // every MMA issued so far has finished before TMEM is released
        mbar_wait_bounded(&drain[wm], 0, nullptr);
      }
    }
  } else {
    // ------------------------------------------------------------------ softmax warpgroups
    const int wg = (warp - 3) >> 2;  // row block 2 * pair + wg
    const int sub = warp & 3;        // TMEM sub-partition of this warp
    const int m = sub * 32 + lane;   // TMEM lane = row of the block
    const int row0 = (2 * pair + wg) * p.rows_per_group;
    const int rows_here = min(p.rows_per_group, p.rows - row0);
    const bool real = m < rows_here;
    const int rr = row0 + m;
    const int jq = real ? rr / p.G : 0;
    const unsigned long long anc = (MASK == kMaskTree && real) ? p.anc[jq] : 0ull;
    const uint32_t tl = tmem + ((uint32_t)(sub * 32) << 16);
    const uint32_t obuf = tl + p_col_o(wg);
    uint8_t* qblock = qs + wg * kPQBlock;
    const float sc = p.scale_log2;

    // all lanes wait, then re-converge (the TMEM accesses that follow are warp-collective)
    auto warp_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
      const bool got = mbar_wait_bounded(bar, parity, &s_abort);
      return __all_sync(0xffffffffu, got);
    };
    auto load_q = [&](int b, int g) {
      p_store_q(p, real, jq, rr, b, g, qblock, m);
      tc::fence_proxy_async_smem();  // the tensor core reads the tile through the async proxy
      __syncwarp();
      if (lane == 0) mbar_arrive(&qfull[wg]);
    };

    Walker w;
    walker_init(p, cta, w);
    int b, g, kb, ke, len;
    bool have = walker_next(p, w, b, g, kb, ke, len);
    if (have && !p.q_tma) load_q(b, g);
    int t = 0, pv_seen = 0;
    bool ok = true;
    while (have && ok) {
      const int n = (ke - kb + kPKeys - 1) / kPKeys;
      int nb = 0, ng = 0, nkb = 0, nke = 0, nlen = 0;
      const bool have_next = walker_next(p, w, nb, ng, nkb, nke, nlen);
      const int tail_start = len - p.nq;
      float m_run = neg_inf(), l = 0.f;
      for (int i = 0; i < n; ++i, ++t) {
        const int key0 = kb + i * kPKeys;
        const uint32_t sbuf = tl + p_col_s(wg, t & 1);
        if (!warp_wait(&sfull[wg][t & 1], (t >> 1) & 1)) { ok = false; break; }
        tc::fence_after();
        // the next part's Q rows into L2 a few tiles ahead (its loads then do not queue behind the
        // K/V stream); once this block's last Q K^T of the part has completed, into shared memory
        if (i == max(n - 4, 0) && have_next && real) {
          const char* a = reinterpret_cast<const char*>(reinterpret_cast<const __nv_bfloat16*>(p.q) +
                                                        (int64_t)nb * p.q_sb + (int64_t)jq * p.q_st +
                                                        (int64_t)(ng * p.G + rr % p.G) * p.q_sh);
          asm volatile("prefetch.global.L2 [%0];" ::"l"(a));
          asm volatile("prefetch.global.L2 [%0];" ::"l"(a + 128));
        }
        if (i == n - 1 && have_next) load_q(nb, ng);
        uint32_t ua[32], ub[32];
        tc::ld32(sbuf, ua);
        tc::ld32(sbuf + 32, ub);
        // keys of this tile the row may see (none for padding rows); the masked path only where
        // some lane of the warp has a hidden key
        const unsigned long long vis =
            real ? p_tile_vis<MASK>(key0, ke, tail_start, jq, anc) : 0ull;
        const bool edge = __any_sync(0xffffffffu, vis != ~0ull);
        const uint32_t vlo = (uint32_t)vis, vhi = (uint32_t)(vis >> 32);
        if (key0 + kPKeys > len) {
          const int s = t % kPStages;
          if (!warp_wait(&full[s], (t / kPStages) & 1)) { ok = false; break; }
          p_zero_v_tail(stages + s * 2 * kPTile + kPTile, key0, len, m);
          tc::fence_proxy_async_smem();
        }
        tc::ld_wait(ua);
        tc::ld_wait(ub);
        // ---- the row's largest visible scaled score in this tile
        float tmax;
        {
          float mx[4] = {neg_inf(), neg_inf(), neg_inf(), neg_inf()};
          if (!edge) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              mx[e & 3] = fmax3(mx[e & 3], __uint_as_float(ua[e]), __uint_as_float(ub[e]));
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              mx[e & 3] = fmaxf(mx[e & 3], (vlo >> e) & 1u ? __uint_as_float(ua[e]) : neg_inf());
              mx[e & 3] = fmaxf(mx[e & 3], (vhi >> e) & 1u ? __uint_as_float(ub[e]) : neg_inf());
            }
          }
          const float raw_max = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
          tmax = (real && raw_max != neg_inf()) ? raw_max * sc : neg_inf();
        }
        // ---- reference max: set by the part's first tile; afterwards moved (with O rescaled) only
        // when the tile max exceeds it by more than 2^8
        if (i == 0) {
          m_run = tmax;
        } else {
          const bool need = tmax > m_run + kPRescaleLog2 || (m_run == neg_inf() && tmax > neg_inf());
          if (__any_sync(0xffffffffu, need)) {
            // O may only be touched once the previous P.V has completed
            if (pv_seen < t) {
              if (!warp_wait(&pvdone[wg][(t - 1) & 1], ((t - 1) >> 1) & 1)) { ok = false; break; }
              pv_seen = t;
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
            for (int c4 = 0; c4 < kPD / 32; ++c4) {
              tc::ld32(obuf + c4 * 32, u);
              tc::ld_wait(u);
#pragma unroll
              for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
              tc::st32(obuf + c4 * 32, u);
            }
            tc::st_wait();
          }
        }
        // ---- P = 2^(s * scale - mu) as bf16 pairs over the buffer's first 32 columns
        {
          const float mu = m_run == neg_inf() ? 0.f : m_run;
          float sums[4] = {0.f, 0.f, 0.f, 0.f};
          auto chunk = [&](const uint32_t (&u)[32], uint32_t vbits, int c2) {
            uint32_t pk[16];
            if (!edge) {
#pragma unroll
              for (int e = 0; e < 32; e += 2) {
                float x0, x1;
                fma2(__uint_as_float(u[e]), __uint_as_float(u[e + 1]), sc, -mu, x0, x1);
                const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                add2(sums[(e >> 1) & 1], sums[2 + ((e >> 1) & 1)], p0, p1);
                pk[e / 2] = pack_bf16(p0, p1);
              }
            } else {
#pragma unroll
              for (int e = 0; e < 32; e += 2) {
                float x0 = fmaf(__uint_as_float(u[e]), sc, -mu);
                float x1 = fmaf(__uint_as_float(u[e + 1]), sc, -mu);
                x0 = (vbits >> e) & 1u ? x0 : neg_inf();
                x1 = (vbits >> (e + 1)) & 1u ? x1 : neg_inf();
                const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                sums[(e >> 1) & 3] += p0 + p1;
                pk[e / 2] = pack_bf16(p0, p1);
              }
            }
            __syncwarp();
            tc::st16(sbuf + c2 * 16, pk);
          };
          chunk(ua, vlo, 0);
          chunk(ub, vhi, 1);
          tc::st_wait();
          l += real ? (sums[0] + sums[1]) + (sums[2] + sums[3]) : 0.f;
        }
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pfull[wg][t & 1]);
      }
      if (!ok) break;
      // ---- epilogue: the part's (m, l, o) record of this row block, once its last P.V is done
      if (pv_seen < t) {
        if (!warp_wait(&pvdone[wg][(t - 1) & 1], ((t - 1) >> 1) & 1)) { ok = false; break; }
        pv_seen = t;
      }
      __syncwarp();
      tc::fence_after();
      {
        // o as a column-major block [D][128 rows] of the part's slot: a warp's store of one column
        // is one 128-byte line
        const int64_t slot = (int64_t)(b * p.Hkv + g) + cta;
        float* blk = p.part_o + (slot * (2 * pairs) + 2 * pair + wg) * (int64_t)(kPD * kPRows) + m;
        uint32_t u[32];
#pragma unroll
        for (int c4 = 0; c4 < kPD / 32; ++c4) {
          __syncwarp();
          tc::ld32(obuf + c4 * 32, u);
          tc::ld_wait(u);
#pragma unroll
          for (int e = 0; e < 32; ++e) blk[(c4 * 32 + e) * kPRows] = __uint_as_float(u[e]);
        }
        if (real) p.part_ml[slot * p.rows + rr] = make_float2(m_run, l);
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ofree[wg]);
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
    tc::dealloc(tmem, kPTmemCols);
  }
}

// Merge of the pair kernel's records: grid (segments, 2 * pairs row blocks, D / 8 column chunks),
// 128 threads, thread m = row m of the block.  The records of a row are read in batches of six
// with all their loads in flight at once: first the (m, l) pairs, then the o columns of the
// column-major blocks (one 128-byte line per column and warp).  Each thread then stores its row's
// 8 columns, one 32-byte chunk of the output row.
constexpr int kMergeCols = 8;
constexpr int kMergeBatch = 6;

__global__ void __launch_bounds__(128) attn_merge_pair(const __grid_constant__ AttnParams p) {
  const int s = blockIdx.x, blk = blockIdx.y, cc = blockIdx.z;
  const int m = threadIdx.x;
  const int b = s / p.Hkv, g = s % p.Hkv;
  const int nblk = 2 * ((p.tc_groups + 1) / 2);
  const int row0 = blk * p.rows_per_group;
  const int rows_here = min(p.rows_per_group, p.rows - row0);
  int64_t total, cum_b;
  warp_scan_tiles(p, b, total, cum_b);
  const int len = seg_len(p, b);
  const bool real = m < rows_here;
  const int rr = row0 + m;
  float acc[kMergeCols];
#pragma unroll
  for (int e = 0; e < kMergeCols; ++e) acc[e] = 0.f;
  // the record positions depend on the lengths only (inputs): worked out above while the partial
  // kernel still runs; its records from here on
  pdl_wait();
  if (len > 0 && real) {
    const int ntiles = seg_tiles(len);
    const int64_t per = tiles_per_cta(p, total);
    const int64_t start = cum_b + (int64_t)g * ntiles;
    const int c0 = (int)(start / per), nrec = (int)((start + ntiles - 1) / per) - c0 + 1;
    const float2* ml_row = p.part_ml + (int64_t)(s + c0) * p.rows + rr;
    const float* o_row = p.part_o + ((int64_t)(s + c0) * nblk + blk) * (int64_t)(kPD * kPRows) +
                         (cc * kMergeCols) * kPRows + m;
    const int64_t rec_stride = (int64_t)nblk * kPD * kPRows;
    float L = 0.f;
    if (nrec <= kMergeBatch) {
      // the usual case: every (m, l) pair and o column of the row in flight at once
      float2 ml[kMergeBatch];
      float v[kMergeBatch][kMergeCols];
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {
        const bool in = u < nrec;
        ml[u] = in ? ml_row[(int64_t)u * p.rows] : make_float2(neg_inf(), 0.f);
#pragma unroll
        for (int e = 0; e < kMergeCols; ++e) v[u][e] = in ? o_row[u * rec_stride + e * kPRows] : 0.f;
      }
      float M = neg_inf();
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) M = fmaxf(M, ml[u].x);
      if (M != neg_inf()) {
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) {
          const float w = ml[u].x == neg_inf() ? 0.f : exp2f(ml[u].x - M);
          L += w * ml[u].y;
#pragma unroll
          for (int e = 0; e < kMergeCols; ++e) acc[e] = fmaf(w, v[u][e], acc[e]);
        }
      }
    } else {
      float M = neg_inf();
      for (int i0 = 0; i0 < nrec; i0 += kMergeBatch) {
        float2 ml[kMergeBatch];
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u)
          ml[u] = i0 + u < nrec ? ml_row[(int64_t)(i0 + u) * p.rows] : make_float2(neg_inf(), 0.f);
#pragma unroll
        for (int u = 0; u < kMergeBatch; ++u) M = fmaxf(M, ml[u].x);
      }
      if (M != neg_inf()) {
        for (int i0 = 0; i0 < nrec; i0 += kMergeBatch) {
          float2 ml[kMergeBatch];
          float v[kMergeBatch][kMergeCols];
#pragma unroll
          for (int u = 0; u < kMergeBatch; ++u) {
            const bool in = i0 + u < nrec;
            ml[u] = in ? ml_row[(int64_t)(i0 + u) * p.rows] : make_float2(neg_inf(), 0.f);
#pragma unroll
            for (int e = 0; e < kMergeCols; ++e) v[u][e] = in ? o_row[(i0 + u) * rec_stride + e * kPRows] : 0.f;
          }
#pragma unroll
          for (int u = 0; u < kMergeBatch; ++u) {
            const float w = ml[u].x == neg_inf() ? 0.f : exp2f(ml[u].x - M);
            L += w * ml[u].y;
#pragma unroll
            for (int e = 0; e < kMergeCols; ++e) acc[e] = fmaf(w, v[u][e], acc[e]);
          }
        }
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
    for (int e = 0; e < kMergeCols; ++e) acc[e] *= inv;
  } else if (len <= 0 && m == 0 && g == 0 && blk == 0 && cc == 0) {
    atomicOr(p.status, p.is_window ? (uint32_t)SPEC_STATUS_BAD_POS : (uint32_t)SPEC_STATUS_BAD_KV_LEN);
  }
  // the row's 8 columns are one 32-byte chunk of the output row: written by this thread
  if (real) {
    const int j = rr / p.G, h = g * p.G + rr % p.G;
    const int64_t off = (int64_t)b * p.o_sb + (int64_t)j * p.o_st + (int64_t)h * p.o_sh + cc * kMergeCols;
    // vector stores where the caller's layout makes the chunk 16-byte aligned, else scalar ones
    if (p.o_bf16) {
      __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.o) + off;
      if ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
        uint4 v;
        v.x = pack_bf16(acc[0], acc[1]);
        v.y = pack_bf16(acc[2], acc[3]);
        v.z = pack_bf16(acc[4], acc[5]);
        v.w = pack_bf16(acc[6], acc[7]);
        *reinterpret_cast<uint4*>(dst) = v;
      } else {
#pragma unroll
        for (int e = 0; e < kMergeCols; ++e) dst[e] = __float2bfloat16_rn(acc[e]);
      }
    } else {
      float* dst = reinterpret_cast<float*>(p.o) + off;
      if ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
        reinterpret_cast<float4*>(dst)[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        reinterpret_cast<float4*>(dst)[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
      } else {
#pragma unroll
        for (int e = 0; e < kMergeCols; ++e) dst[e] = acc[e];
      }
    }
  }
}

cudaError_t launch_merge_pair(const AttnParams& p, cudaStream_t stream) {
  if (p.D != kPD || p.nks != 1 || p.has_new) return cudaErrorInvalidValue;
  const dim3 grid(p.B * p.Hkv, 2 * ((p.tc_groups + 1) / 2), kPD / kMergeCols);
  return launch_dependent(attn_merge_pair, grid, dim3(128), 0, stream, 0u, p);
}

template <int MASK>
static cudaError_t launch_pair_mask(const AttnParams& p, const CUtensorMap* tmK, const CUtensorMap* tmV,
                                    const CUtensorMap* tmQ, cudaStream_t stream) {
  const size_t smem = attn_tc_pair_smem_bytes();
  auto kern = attn_partial_tc_pair<MASK>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<p.grid_x * ((p.tc_groups + 1) / 2), kPThreads, smem, stream>>>(*tmK, *tmV, *tmQ, p);
  return cudaGetLastError();
}

cudaError_t launch_partial_tc_pair(const AttnParams& p, const CUtensorMap* tmK, const CUtensorMap* tmV,
                                   const CUtensorMap* tmQ, cudaStream_t stream) {
  if (p.nks != 1 || p.tc_groups < 2) return cudaErrorInvalidValue;
  switch (p.mask) {
    case kMaskNone: return launch_pair_mask<kMaskNone>(p, tmK, tmV, tmQ, stream);
    case kMaskChain: return launch_pair_mask<kMaskChain>(p, tmK, tmV, tmQ, stream);
    default: return launch_pair_mask<kMaskTree>(p, tmK, tmV, tmQ, stream);
  }
}

}  // namespace specv
