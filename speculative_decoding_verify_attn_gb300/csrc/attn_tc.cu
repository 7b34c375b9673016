// Split-KV verify attention on the 5th-generation tensor core, for query blocks dense enough to
// be a real contraction (nq * G > 32 rows per kv head: the 70B-shaped chain with 7 x 8 = 56 rows,
// Medusa-style trees with 64 x 4 = 256 rows).
//
// Same stream-K decomposition, workspace records and merge kernel as the mma.sync path (attn.cu);
// one CTA per SM.  Per CTA, one 128-row block of query rows (a "row group"), warp-specialised:
//   warp 0     TMA producer: 128-key K and V tiles (128-byte swizzle) into a 3-stage ring.
//   warp 1     MMA issuer (one lane) and TMEM owner: S = Q K^T (M = 128, N = 128 keys, K = 128)
//              into one of two TMEM score buffers, then O += P V (P read from TMEM, V as an
//              MN-major shared-memory operand) into the TMEM output accumulator.
//   warps 2-5  softmax and epilogue, one thread per TMEM lane (query row): scores from TMEM,
//              masks, online softmax in the log2 domain with lazy rescaling: P is computed in
//              one pass against the running max, and only when a row's max grows by more than
//              2^8 is O rescaled in TMEM and the tile redone; P as bf16 pairs into TMEM; at the
//              end of each part, O and (m, l) to the workspace.
// Query rows are spread over the four TMEM sub-partitions (row r -> lane 32 (r mod 4) + r / 4)
// so that a 56-row block keeps all four softmax warps busy.
// TMEM columns (512 allocated): S buffers [0,128) and [128,256), O [256,384), P (bf16 pairs)
// buffers [384,448) and [448,512).  P has its own columns so that a tile whose running max
// jumps can be redone from its scores.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "attn_common.cuh"
#include "attn_internal.h"
#include "common.cuh"
#include "tcgen05.cuh"

namespace specv {

constexpr int kTcRows = 128;     // M: query rows per CTA
constexpr int kTcKeys = 128;     // keys per tile (N of QK^T, K of PV)
constexpr int kTcStages = 3;
constexpr int kTcD = 128;
constexpr uint32_t kTmemCols = 512;
constexpr int kTcThreads = 192;  // TMA warp, MMA warp, 4 softmax warps
constexpr int kTile = kTcKeys * kTcD * 2;   // bytes of one K (or V) tile: 32 KB
constexpr int kHalf = kTcKeys * 128;        // one 64-column (128-byte) half of a tile: 16 KB
constexpr int kQHalf = kTcRows * 128;       // one half of the Q block: 16 KB
constexpr float kRescaleLog2 = 8.0f;        // lazy-rescale threshold: 2^8
constexpr uint32_t kColO = 2 * kTcKeys;     // TMEM column of the O accumulator
constexpr uint32_t kColP = 3 * kTcKeys;     // TMEM column of P buffer 0 (buffer 1 at +64)

constexpr uint32_t kIdescQK = tc::idesc_bf16(kTcRows, kTcKeys, 0, 0);  // A = Q (K-major), B = K (K-major)
constexpr uint32_t kIdescPV = tc::idesc_bf16(kTcRows, kTcD, 0, 1);     // A = P (TMEM), B = V (MN-major)

size_t attn_tc_smem_bytes() { return 1024 + (size_t)kTcStages * 2 * kTile + 2 * (size_t)kQHalf; }

__device__ __forceinline__ int tc_row_of_lane(int m) { return 4 * (m & 31) + (m >> 5); }

template <int MASK>
__global__ void __launch_bounds__(kTcThreads, 1)
    attn_partial_tc(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[kTcStages], empty[kTcStages], sfull[2], pfull[2];
  __shared__ uint64_t pvdone, qfull, ofree, drain;
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
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sfull[i], 1);
      mbar_init(&pfull[i], 4);
    }
    mbar_init(&pvdone, 1);
    mbar_init(&qfull, 4);
    mbar_init(&ofree, 4);
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
    atomicOr(p.status, (uint32_t)SPEC_STATUS_TIMEOUT);
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
      while (ok && walker_next(p, w, b, g, kb, ke, len)) {
        for (int key0 = kb; key0 < ke; key0 += kTcKeys, ++t) {
          const int s = t % kTcStages;
          if (!mbar_wait_bounded(&empty[s], ((t / kTcStages) & 1) ^ 1u, &s_abort)) {
            fail();
            ok = false;
            break;
          }
          uint8_t* sk = stages + s * 2 * kTile;
          mbar_arrive_expect_tx(&full[s], 2u * kTile);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            tma_load_4d(sk + h * kHalf, &tmK, &full[s], h * 64, key0, g, b);
            tma_load_4d(sk + kTile + h * kHalf, &tmV, &full[s], h * 64, key0, g, b);
          }
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
    Walker w;
    walker_init(p, cta, w);
    if (lane == 0) {
      int t = 0, part = 0;
      bool ok = true;
      int prev_t = -1, prev_first = 0, prev_part = 0;
      auto issue_pv = [&](int tt, int first, int pt) -> bool {
        if (first && pt >= 1 && !mbar_wait_bounded(&ofree, (pt - 1) & 1, &s_abort)) return false;
        if (!mbar_wait_bounded(&pfull[tt & 1], (tt >> 1) & 1, &s_abort)) return false;
        tc::fence_after();
        const uint32_t vb = stages_u32 + (tt % kTcStages) * 2 * kTile + kTile;
        const uint32_t pa = tmem + kColP + (uint32_t)(tt & 1) * (kTcKeys / 2);
#pragma unroll
        for (int ks = 0; ks < kTcKeys / 16; ++ks) {
          const uint64_t bdesc = tc::smem_desc(vb + ks * 2048, kHalf, 1024);
          tc::mma_ts(tmem + kColO, pa + ks * 8, bdesc, kIdescPV, (ks > 0 || !first) ? 1u : 0u);
        }
        tc::commit(&pvdone);
        tc::commit(&empty[tt % kTcStages]);
        return true;
      };
      int b, g, kb, ke, len;
      while (ok && walker_next(p, w, b, g, kb, ke, len)) {
        for (int key0 = kb; key0 < ke; key0 += kTcKeys, ++t) {
          const int first = key0 == kb;
          if (first && !mbar_wait_bounded(&qfull, part & 1, &s_abort)) { ok = false; break; }
          const int s = t % kTcStages;
          if (!mbar_wait_bounded(&full[s], (t / kTcStages) & 1, &s_abort)) { ok = false; break; }
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
          if (prev_t >= 0 && !issue_pv(prev_t, prev_first, prev_part)) { ok = false; break; }
          prev_t = t;
          prev_first = first;
          prev_part = part;
        }
        ++part;
      }
      if (ok && prev_t >= 0 && !issue_pv(prev_t, prev_first, prev_part)) ok = false;
      if (!ok) {
        fail();
        tc::commit(&drain);  // every MMA issued so far has finished before TMEM is released
        mbar_wait_bounded(&drain, 0, nullptr);
      }
    }
  } else {
    // ------------------------------------------------------------------ softmax + epilogue
    const int sub = warp & 3;                      // TMEM sub-partition of this warp
    const int m = sub * 32 + lane;                 // TMEM lane = M row
    const int r = tc_row_of_lane(m);               // query row within the row group
    const bool real = r < rows_here;
    const int rr = row0 + r;
    const int jq = real ? rr / p.G : 0;            // query position (chain row / tree node)
    const unsigned long long anc = (MASK == kMaskTree && real) ? p.anc[jq] : 0ull;
    const uint32_t tl = tmem + ((uint32_t)(sub * 32) << 16);
    const __nv_bfloat16* qbase = reinterpret_cast<const __nv_bfloat16*>(p.q);
    const int stid = threadIdx.x - 64;             // 0..127 over the softmax warps

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
    if (have) load_q(b, g);
    int t = 0, pv_seen = 0;
    bool ok = true;
    while (have && ok) {
      float m_used = neg_inf(), l = 0.f;
      const int tail_start = len - p.nq;
      for (int key0 = kb; key0 < ke; key0 += kTcKeys, ++t) {
        if (!warp_wait(&sfull[t & 1], (t >> 1) & 1)) { ok = false; break; }
        tc::fence_after();
        const bool edge = key0 + kTcKeys > ke || (MASK != kMaskNone && key0 + kTcKeys > tail_start);
        const uint32_t sbuf = tl + (uint32_t)(t & 1) * kTcKeys;
        const uint32_t pbuf = tl + kColP + (uint32_t)(t & 1) * (kTcKeys / 2);
        const float sc = p.scale_log2;
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
        // P = 2^(score * scale - mu) for the whole tile, as bf16 pairs in this tile's P buffer
        // (chunk c4 of 32 keys in columns [16 c4, 16 c4 + 16)); the scores stay untouched.
        // Returns the row's sum of P and the largest visible (score * scale - mu).
        // tcgen05.ld/st are warp-collective: every lane runs this, padding rows included; the
        // inner loops are branch-free (masked keys become -inf, and 2^-inf = 0).
        auto p_pass = [&](float mu, float& sum_out, float& xmax_out) {
          float sums[4] = {0.f, 0.f, 0.f, 0.f};
          float xm[4] = {neg_inf(), neg_inf(), neg_inf(), neg_inf()};
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            uint32_t u[32], pk[16];
            tc::ld32(sbuf + c4 * 32, u);
            tc::ld_wait();
            if (!edge) {
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                const float x0 = fmaf(__uint_as_float(u[i]), sc, -mu);
                const float x1 = fmaf(__uint_as_float(u[i + 1]), sc, -mu);
                xm[(i >> 1) & 3] = fmaxf(xm[(i >> 1) & 3], fmaxf(x0, x1));
                const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                sums[(i >> 1) & 3] += p0 + p1;
                pk[i / 2] = pack_bf16(p0, p1);
              }
            } else {
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                const int kk = key0 + c4 * 32 + i;
                float x0 = fmaf(__uint_as_float(u[i]), sc, -mu);
                float x1 = fmaf(__uint_as_float(u[i + 1]), sc, -mu);
                x0 = (real & key_visible_nb<MASK>(kk, ke, tail_start, jq, anc)) ? x0 : neg_inf();
                x1 = (real & key_visible_nb<MASK>(kk + 1, ke, tail_start, jq, anc)) ? x1 : neg_inf();
                xm[(i >> 1) & 3] = fmaxf(xm[(i >> 1) & 3], fmaxf(x0, x1));
                const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                sums[(i >> 1) & 3] += p0 + p1;
                pk[i / 2] = pack_bf16(p0, p1);
              }
            }
            __syncwarp();
            tc::st16(pbuf + c4 * 16, pk);
          }
          tc::st_wait();
          sum_out = (sums[0] + sums[1]) + (sums[2] + sums[3]);
          xmax_out = real ? fmaxf(fmaxf(xm[0], xm[1]), fmaxf(xm[2], xm[3])) : neg_inf();
        };
        auto rescale_o = [&](float alpha) {  // O row *= alpha (warp-collective)
          uint32_t u[32];
#pragma unroll 1
          for (int c4 = 0; c4 < 4; ++c4) {
            const uint32_t oa = tl + kColO + c4 * 32;
            tc::ld32(oa, u);
            tc::ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
            tc::st32(oa, u);
          }
          tc::st_wait();
        };
        float sum = 0.f, xmax = neg_inf();
        const bool first = key0 == kb;
        if (first) {
          // first tile of a part: the row max first, then P against it
          float mx[4] = {neg_inf(), neg_inf(), neg_inf(), neg_inf()};
          uint32_t u[32];
#pragma unroll 1
          for (int c4 = 0; c4 < 4; ++c4) {
            tc::ld32(sbuf + c4 * 32, u);
            tc::ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              float x = __uint_as_float(u[i]) * sc;
              if (edge) x = key_visible_nb<MASK>(key0 + c4 * 32 + i, ke, tail_start, jq, anc) ? x : neg_inf();
              mx[i & 3] = fmaxf(mx[i & 3], x);
            }
          }
          m_used = real ? fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) : neg_inf();
          __syncwarp();
        }
        // Later tiles: P against the running max in one pass; only if some row's max grew by more
        // than 2^8 (or the row had seen nothing yet) is O rescaled and the tile redone once.
#pragma unroll 1
        for (int attempt = 0; attempt < 2; ++attempt) {
          const float mu = m_used == neg_inf() ? 0.f : m_used;
          p_pass(mu, sum, xmax);
          if (first || attempt == 1) break;
          const bool need = real && (xmax > kRescaleLog2 || (m_used == neg_inf() && xmax > neg_inf()));
          if (!__any_sync(0xffffffffu, need)) break;
          // O may only be touched once the previous tile's P.V has completed (every P.V completion
          // is observed exactly once, in order)
          if (t >= 1 && pv_seen == t - 1) {
            if (!warp_wait(&pvdone, (t - 1) & 1)) { ok = false; break; }
            pv_seen = t;
            tc::fence_after();
          }
          float alpha = 1.f;
          if (need) {
            const float m_new = xmax + mu;
            alpha = (m_used == neg_inf()) ? 0.f : ex2_approx(m_used - m_new);
            l *= alpha;
            m_used = m_new;
          }
          __syncwarp();
          rescale_o(alpha);
          __syncwarp();
        }
        if (!ok) break;
        l += real ? sum : 0.f;
        // observe the previous tile's P.V completion (if the rescale path did not) before this
        // tile's P is handed over, so that the P.V barrier never runs two phases ahead
        if (t >= 1 && pv_seen == t - 1) {
          if (!warp_wait(&pvdone, (t - 1) & 1)) { ok = false; break; }
          pv_seen = t;
        }
        tc::fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pfull[t & 1]);
      }
      if (!ok) break;
      // next part's Q: every Q K^T of this part has completed (its last scores were read)
      const int cb = b, cg = g;
      have = walker_next(p, w, b, g, kb, ke, len);
      if (have) load_q(b, g);
      // epilogue: O of this part once its last P.V has completed
      if (pv_seen == t - 1) {
        if (!warp_wait(&pvdone, (t - 1) & 1)) { ok = false; break; }
        pv_seen = t;
      }
      __syncwarp();
      tc::fence_after();
      {
        const int64_t slot = (int64_t)(cb * p.Hkv + cg) + cta;
        const int64_t rec = slot * p.rows + rr;
        uint32_t u[32];
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          __syncwarp();
          tc::ld32(tl + kColO + c4 * 32, u);
          tc::ld_wait();
          if (real) {
            float4* dst = reinterpret_cast<float4*>(p.part_o + rec * kTcD + c4 * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(u[4 * i]), __uint_as_float(u[4 * i + 1]),
                                   __uint_as_float(u[4 * i + 2]), __uint_as_float(u[4 * i + 3]));
          }
        }
        if (real) p.part_ml[rec] = make_float2(m_used, l);
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ofree);
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
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<p.grid_x * p.tc_groups, kTcThreads, smem, stream>>>(*tmK, *tmV, p);
  return cudaGetLastError();
}

cudaError_t launch_partial_tc(const AttnParams& p, const CUtensorMap* tmK, const CUtensorMap* tmV,
                              cudaStream_t stream) {
  switch (p.mask) {
    case kMaskNone: return launch_tc_mask<kMaskNone>(p, tmK, tmV, stream);
    case kMaskChain: return launch_tc_mask<kMaskChain>(p, tmK, tmV, stream);
    default: return launch_tc_mask<kMaskTree>(p, tmK, tmV, stream);
  }
}

}  // namespace specv
