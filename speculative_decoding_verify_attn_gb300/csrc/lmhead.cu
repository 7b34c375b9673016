// The LM-head projection fused with verification (spec_lmhead_sample): the verified rows' logits
// are the target's final hidden states times the LM-head matrix ("Speculative Decoding in LLM
// Serving Systems", The algorithm; "Guide to MagicDec", Implementation Step 3).  The greedy rules
// only need each row's argmax, so there the logits never leave the SM: a tcgen05 GEMM reduces its
// accumulators straight to one 64-bit (value, id) key per hidden row, and a small kernel reads the
// keys and applies the chain or tree rule.  The stochastic rules need whole normalised rows: the
// same GEMM then stores its accumulators as fp32 logits, and the sampling kernels follow.
//
// GEMM (D[v, n] = sum_k W[v, k] H[n, k]): the vocabulary is M (128 rows of W per tile, K-major,
// 128-byte swizzle), the B*R hidden rows are N (padded to a multiple of 16, at most 256).  A CTA
// owns a run of vocabulary tiles and keeps as many accumulators as fit in TMEM (512 / N columns)
// at once, so each 64-element chunk of the hidden rows is staged once per pass for all of them.
// The weight is read exactly once; the run is HBM-bound, so shared memory goes to as deep a
// weight ring as fits beside the hidden-row ring:
//   warp 0     weight producer: each tile's 128-row chunks into a ring of multi-chunk copies.
//   warp 1     MMA issuer (one lane) and TMEM owner: 4 MMAs (K = 16) per weight chunk, a tile
//              taking several K chunks in a row (one accumulator chain; see lmhead_layout).
//   warps 2-5, 7-10  epilogue, two warps per TMEM lane quadrant, taking alternate 32-column
//              blocks of the pass's accumulators (32 hidden rows x the warp's 32 vocabulary rows
//              of every tile): each lane's maximum over the tiles, then two warp reductions per
//              column (the maximum, then the smallest id reaching it; entries past V excluded)
//              give one key per hidden row, merged into the CTA's keys in shared memory; at the
//              end one 64-bit atomic max per row and CTA into global memory.
//   warp 6     hidden-row producer: each pass's K chunks into their own ring.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <limits.h>

#include "common.cuh"
#include "lmhead_internal.h"
#include "spec_verify.h"
#include "tcgen05.cuh"
#include "launch_cache.h"

namespace specv {

constexpr int kLmThreads = 352;               // 11 warps: producers, issuer, 8 epilogue warps
constexpr int kLmEpiWarps = 8;
constexpr int kLmWChunk = 128 * 128;          // bytes: 128 vocabulary rows x 64 bf16
constexpr int kLmSmemCap = 227 * 1024;        // dynamic shared memory of one CTA
constexpr int kLmWStagesMax = 16;
constexpr int kLmHStagesMax = 8;

// Ring layout.  A tile takes `kgroup` K chunks in a row, so its accumulator sees chains of
// 4 kgroup MMAs: on GB300 a chain of 4 small-N MMAs costs about 660 cycles, of 16 about 1300, so
// chains of 4 would leave the single issuer slower than the weight stream; the group is 4 chunks
// where the hidden rows are few (npad <= 96) and 2 otherwise.  Both rings take several K chunks
// per copy (3-D boxes): an SM's tensor-memory-access unit completes copies at a rate set more by
// their number than by their size (about one per 0.3 us for 16-32 KB boxes), so 16 KB copies
// alone would cap an SM near the HBM share it needs for the weight, and the hidden rows' copies
// on top of those slow the weight stream down.  The hidden ring holds two groups (the one in use
// and the next) in one copy each; the rest of shared memory is weight, two chunks per copy (at
// 256 rows only two copies, which measured faster than three one-chunk hidden copies beside three
// weight copies).
LmLayout lmhead_layout(int npad) {
  LmLayout L;
  const size_t budget = kLmSmemCap - 1024 - 2560;  // alignment pad; static barriers and keys
  L.kgroup = npad <= 96 ? 4 : 2;
  L.wbox = 2;
  L.hbox = L.kgroup;
  L.h_stages = 2;
  const size_t hb = (size_t)npad * 128 * L.hbox, wb = (size_t)kLmWChunk * L.wbox;
  int ws = (int)((budget - L.h_stages * hb) / wb);
  L.w_stages = ws > kLmWStagesMax ? kLmWStagesMax : ws;
  L.smem = 1024 + (size_t)L.w_stages * wb + (size_t)L.h_stages * hb;
  return L;
}

// Keys: (ord(value) << 32) | ~id, so that the unsigned order is: larger value first, then smaller id.
__device__ __forceinline__ int lm_key_id(unsigned long long k) { return (int)(~(uint32_t)k); }

// The steps of a CTA's run of vocabulary tiles: passes of up to `tpp` tiles; per pass, per group
// of kgroup K chunks, per tile of the pass, the group's weight chunks of that tile.
struct LmWalk {
  int tile0, ntiles, tpp, nk;
};
__device__ __forceinline__ LmWalk lm_walk(const LmheadParams& p) {
  LmWalk w;
  const int per = (p.n_vtiles + gridDim.x - 1) / gridDim.x;
  w.tile0 = min((int)blockIdx.x * per, p.n_vtiles);
  w.ntiles = min(per, p.n_vtiles - w.tile0);
  w.tpp = p.tiles_per_pass;
  w.nk = p.d / 64;
  return w;
}

// One box of a [rows, d] bf16 matrix viewed as (column in chunk, row, chunk): `box chunks` K
// chunks of 64 columns of the box's rows, landing chunk after chunk ([chunk][row][128 B]).
__device__ __forceinline__ void lm_tma_load_chunks(void* smem_dst, const void* tmap, uint64_t* bar, int row0,
                                                   int chunk0) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(0), "r"(row0), "r"(chunk0), "r"(smem_u32(bar))
      : "memory");
}
// Whole warp: 16 consecutive 32-bit TMEM columns of this warp's 32 lanes, waited for in the same
// statement (the registers are valid once it returns).
__device__ __forceinline__ void lm_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
// Monotone map of fp32 to u32 (a < b  <=>  ord(a) < ord(b), a == b  <=>  ord(a) == ord(b) for
// non-NaN values: -0 is taken as +0, so a zero maximum still ties to the smaller id); 0 lies below
// every mapped value and stands for "no entry".
__device__ __forceinline__ uint32_t lm_ord(float v) {
  uint32_t u = __float_as_uint(v);
  if ((u << 1) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// Warp reductions as compiler intrinsics (not volatile asm), so that the reductions of different
// columns can overlap instead of each waiting for the one before it.
__device__ __forceinline__ uint32_t lm_redux_max(uint32_t x) { return __reduce_max_sync(0xffffffffu, x); }
__device__ __forceinline__ uint32_t lm_redux_min(uint32_t x) { return __reduce_min_sync(0xffffffffu, x); }
__device__ __forceinline__ void lm_epi_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kLmEpiWarps * 32) : "memory"); }

// NC consecutive accumulator columns (hidden rows) starting at TMEM address `col0` of tile 0, over
// the pass's nt tiles (tile t at column offset t * npad; this lane's vocabulary id vm0 + 128 t):
// first each lane's own maximum over the tiles (earlier tile first, so equal values keep the
// smaller id; ids >= V excluded), then per column the warp's maximum and the smallest id reaching
// it.  Lane e keeps column e's pair in (bo, bi).
template <int NC>
__device__ __forceinline__ void lm_reduce_tiles(uint32_t col0, int npad, int nt, uint32_t vm0, uint32_t V, int lane,
                                                uint32_t& bo, uint32_t& bi) {
  uint32_t o[NC], ix[NC];
#pragma unroll
  for (int e = 0; e < NC; ++e) {
    o[e] = 0u;
    ix[e] = 0xffffffffu;
  }
  for (int t = 0; t < nt; ++t) {
    uint32_t u[32];
    if constexpr (NC == 32) {
      tc::ld32(col0 + (uint32_t)(t * npad), u);
      tc::ld_wait(u);
    } else {
      lm_ld16(col0 + (uint32_t)(t * npad), *reinterpret_cast<uint32_t(*)[16]>(u));
    }
    const uint32_t vm = vm0 + 128u * (uint32_t)t;
    const bool valid = vm < V;
#pragma unroll
    for (int e = 0; e < NC; ++e) {
      const uint32_t x = valid ? lm_ord(__uint_as_float(u[e])) : 0u;
      if (x > o[e]) {
        o[e] = x;
        ix[e] = vm;
      }
    }
  }
  uint32_t mo[NC];
#pragma unroll
  for (int e = 0; e < NC; ++e) mo[e] = lm_redux_max(o[e]);
#pragma unroll
  for (int e = 0; e < NC; ++e) {
    const uint32_t mi = lm_redux_min(o[e] == mo[e] ? ix[e] : 0xffffffffu);
    if (lane == e) {
      bo = mo[e];
      bi = mi;
    }
  }
}

// STORE: write the fp32 logits [nrows][V] instead of reducing them to argmax keys (stochastic
// modes); for a fixed hidden row a warp's 32 lanes hold 32 consecutive vocabulary rows, so each
// column of a TMEM load is one 128-byte store.
template <bool STORE>
__global__ void __launch_bounds__(kLmThreads, 1)
    lmhead_gemm(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmH,
                const __grid_constant__ LmheadParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t wfull[kLmWStagesMax], wempty[kLmWStagesMax], hfull[kLmHStagesMax], hempty[kLmHStagesMax];
  __shared__ uint64_t acc_full, acc_empty, drain;
  __shared__ uint32_t tmem_base;
  __shared__ int s_abort;
  __shared__ unsigned long long s_key[kLmMaxRows];   // this CTA's running key per hidden row
  const uint32_t raw = smem_u32(smem_raw);
  const int WS = p.w_stages, HS = p.h_stages, WB = p.wbox, HB = p.hbox;
  const int wslot = WB * kLmWChunk;                                 // one weight copy: WB chunks
  const int hchunk = p.npad * 128;                                  // one hidden chunk, 1 KB multiple
  const int hslot = HB * hchunk;                                    // one hidden copy: HB chunks
  uint8_t* wring = smem_raw + (((raw + 1023u) & ~1023u) - raw);     // [slot][chunk][128 rows][128 B]
  uint8_t* hring = wring + WS * wslot;                              // [slot][chunk][npad rows][128 B]
  const uint32_t wring_u32 = smem_u32(wring), hring_u32 = smem_u32(hring);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const LmWalk W = lm_walk(p);
  const int npass = (W.ntiles + W.tpp - 1) / W.tpp;

  if (threadIdx.x == 0) {
    for (int i = 0; i < WS; ++i) {
      mbar_init(&wfull[i], 1);
      mbar_init(&wempty[i], 1);
    }
    for (int i = 0; i < HS; ++i) {
      mbar_init(&hfull[i], 1);
      mbar_init(&hempty[i], 1);
    }
    mbar_init(&acc_full, 1);
    mbar_init(&acc_empty, kLmEpiWarps);
    mbar_init(&drain, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  for (int r = threadIdx.x; r < kLmMaxRows; r += blockDim.x) s_key[r] = 0ull;
  if (warp == 1) tc::alloc(&tmem_base, 512);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = tmem_base;
  auto fail = [&]() {
    s_abort = 1;
    atomicOr(p.status, (uint32_t)SPEC_STATUS_TIMEOUT);
  };

  // Copies per group of gk chunks: ceil(gk / box) (a last group shorter than the box reads
  // chunks past d, which the copy fills with zeros and no MMA reads).
  if (warp == 0) {
    // ------------------------------------------------------------------ weight producer
    if (lane == 0 && W.ntiles > 0) {
      tma_prefetch_desc(&tmW);
      int wc = 0;
      bool ok = true;
      for (int p0 = 0; ok && p0 < W.ntiles; p0 += W.tpp) {
        const int nt = min(W.tpp, W.ntiles - p0);
        for (int kg = 0; ok && kg < W.nk; kg += p.kgroup) {
          const int nb = (min(p.kgroup, W.nk - kg) + WB - 1) / WB;
          for (int t = 0; ok && t < nt; ++t) {
            for (int i = 0; i < nb; ++i, ++wc) {
              const int ws = wc % WS;
              if (!mbar_wait_bounded(&wempty[ws], ((wc / WS) & 1) ^ 1u, &s_abort)) { ok = false; break; }
              mbar_arrive_expect_tx(&wfull[ws], (uint32_t)wslot);
              lm_tma_load_chunks(wring + ws * wslot, &tmW, &wfull[ws], (W.tile0 + p0 + t) * 128, kg + i * WB);
            }
          }
        }
      }
      if (!ok) {
        fail();
        for (int i = 1; i <= min(wc, WS); ++i) mbar_wait_bounded(&wfull[(wc - i) % WS], ((wc - i) / WS) & 1, nullptr);
      }
    }
  } else if (warp == 6) {
    // ------------------------------------------------------------------ hidden-row producer
    if (lane == 0 && W.ntiles > 0) {
      tma_prefetch_desc(&tmH);
      int hc = 0;
      bool ok = true;
      for (int ps = 0; ok && ps < npass; ++ps) {
        for (int kg = 0; ok && kg < W.nk; kg += p.kgroup) {
          const int nb = (min(p.kgroup, W.nk - kg) + HB - 1) / HB;
          for (int i = 0; i < nb; ++i, ++hc) {
            const int hs = hc % HS;
            if (!mbar_wait_bounded(&hempty[hs], ((hc / HS) & 1) ^ 1u, &s_abort)) { ok = false; break; }
            mbar_arrive_expect_tx(&hfull[hs], (uint32_t)hslot);
            lm_tma_load_chunks(hring + hs * hslot, &tmH, &hfull[hs], 0, kg + i * HB);
          }
        }
      }
      if (!ok) {
        fail();
        for (int i = 1; i <= min(hc, HS); ++i) mbar_wait_bounded(&hfull[(hc - i) % HS], ((hc - i) / HS) & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // One thread issues every MMA, so its instruction stream between MMAs sets the MMA rate: ring
    // slots and phases advance incrementally and descriptors are precomputed (a K step of 16 is
    // +2 in the descriptor's address field, a weight chunk +1024, a hidden chunk +hchunk / 16).
    if (lane == 0 && W.ntiles > 0) {
      const uint32_t idesc = tc::idesc_bf16(128, p.npad, 0, 0);
      const uint64_t ad0 = tc::smem_desc(wring_u32, 16, 1024);
      const uint64_t bd0 = tc::smem_desc(hring_u32, 16, 1024);
      const uint32_t hstep = (uint32_t)hchunk >> 4;
      int ws = 0, hs = 0;
      uint32_t wph = 0, hph = 0;
      bool ok = true;
      for (int ps = 0; ok && ps < npass; ++ps) {
        const int nt = min(W.tpp, W.ntiles - ps * W.tpp);
        if (ps > 0 && !mbar_wait_bounded(&acc_empty, (ps - 1) & 1, &s_abort)) { ok = false; break; }
        for (int kg = 0; ok && kg < W.nk; kg += p.kgroup) {
          const int gk = min(p.kgroup, W.nk - kg);
          const int nwb = (gk + WB - 1) / WB, nhb = (gk + HB - 1) / HB;
          for (int j = 0, s2 = hs, ph = hph; j < nhb; ++j) {
            if (!mbar_wait_bounded(&hfull[s2], ph, &s_abort)) { ok = false; break; }
            if (++s2 == HS) { s2 = 0; ph ^= 1; }
          }
          if (!ok) break;
          tc::fence_after();
          uint32_t tacc = tmem;
          // tile by tile, each taking the group's gk chunks as one chain on its accumulator; the
          // chain's weight copies are released together after it
          for (int t = 0; t < nt; ++t, tacc += (uint32_t)p.npad) {
            for (int j = 0, s2 = ws, ph = wph; j < nwb; ++j) {
              if (!mbar_wait_bounded(&wfull[s2], ph, &s_abort)) { ok = false; break; }
              if (++s2 == WS) { s2 = 0; ph ^= 1; }
            }
            if (!ok) break;
            tc::fence_after();
            for (int j = 0, sw = ws, cw = 0, sh = hs, ch = 0; j < gk; ++j) {
              const uint64_t ad = ad0 + (uint64_t)(sw * (wslot >> 4) + cw * (kLmWChunk >> 4));
              const uint64_t bd = bd0 + (uint64_t)(sh * (hslot >> 4) + ch * hstep);
              tc::mma_ss(tacc, ad, bd, idesc, (kg + j) ? 1u : 0u);
              tc::mma_ss(tacc, ad + 2, bd + 2, idesc, 1u);
              tc::mma_ss(tacc, ad + 4, bd + 4, idesc, 1u);
              tc::mma_ss(tacc, ad + 6, bd + 6, idesc, 1u);
              if (++cw == WB) { cw = 0; if (++sw == WS) sw = 0; }
              if (++ch == HB) { ch = 0; if (++sh == HS) sh = 0; }
            }
            for (int j = 0; j < nwb; ++j) {
              tc::commit(&wempty[ws]);
              if (++ws == WS) { ws = 0; wph ^= 1; }
            }
          }
          if (!ok) break;
          for (int j = 0; j < nhb; ++j) {
            tc::commit(&hempty[hs]);
            if (++hs == HS) { hs = 0; hph ^= 1; }
          }
        }
        if (ok) tc::commit(&acc_full);
      }
      if (!ok) {
        fail();
        tc::commit(&drain);
        mbar_wait_bounded(&drain, 0, nullptr);
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue (warps 2-5, 7-10)
    const int sub = warp & 3;           // TMEM lanes 32 sub .. 32 sub + 31 = vocabulary rows
    const int half = warp >= 7 ? 1 : 0; // the 32-column blocks this warp takes: half, half + 2, ...
    const int eidx = (warp - 2 - half) * 32 + lane;   // 0 .. 255 over the epilogue threads
    for (int ps = 0; ps < npass; ++ps) {
      const int nt = min(W.tpp, W.ntiles - ps * W.tpp);
      const bool got = __all_sync(0xffffffffu, mbar_wait_bounded(&acc_full, ps & 1, &s_abort));
      if (!got) {
        if (lane == 0) fail();
        break;
      }
      tc::fence_after();
      const uint32_t vm0 = (uint32_t)((W.tile0 + ps * W.tpp) * 128 + sub * 32 + lane);  // tile 0's vocabulary id
      const uint32_t tb = tmem + ((uint32_t)(sub * 32) << 16);
      if constexpr (STORE) {
        for (int t = 0; t < nt; ++t) {
          const uint32_t vm = vm0 + 128u * (uint32_t)t;
          for (int cc = half; cc * 32 < p.npad; cc += 2) {
            uint32_t u[32];
            if (cc * 32 + 32 <= p.npad) {
              tc::ld32(tb + (uint32_t)(t * p.npad + cc * 32), u);
              tc::ld_wait(u);
            } else {
              lm_ld16(tb + (uint32_t)(t * p.npad + cc * 32), *reinterpret_cast<uint32_t(*)[16]>(u));
            }
            const int nc = min(32, p.npad - cc * 32);
            if (vm < (uint32_t)p.V) {
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                const int n = cc * 32 + e;
                if (e < nc && n < p.nrows) p.logits[(int64_t)n * p.V + vm] = __uint_as_float(u[e]);
              }
            }
          }
        }
      } else {
        // one 32-column block at a time, not unrolled: the unrolled blocks made a straight run of
        // tens of KB of code executed once per pass, whose instruction fetches set the pace; the
        // block's keys go straight into the CTA's shared keys
#pragma unroll 1
        for (int cc = half; cc * 32 < p.npad; cc += 2) {
          uint32_t bo = 0, bi = 0xffffffffu;
          if (cc * 32 + 32 <= p.npad)
            lm_reduce_tiles<32>(tb + cc * 32, p.npad, nt, vm0, (uint32_t)p.V, lane, bo, bi);
          else
            lm_reduce_tiles<16>(tb + cc * 32, p.npad, nt, vm0, (uint32_t)p.V, lane, bo, bi);
          const int row = cc * 32 + lane;
          if (row < p.nrows && bi < (uint32_t)p.V)
            atomicMax(&s_key[row], ((unsigned long long)bo << 32) | (uint32_t)~bi);
        }
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty);
    }
    if constexpr (!STORE) {
      // the CTA's keys (the epilogue warps met in shared memory), one global atomic per row
      lm_epi_sync();
      unsigned long long* keys = reinterpret_cast<unsigned long long*>(p.rec);
      for (int r = eidx; r < p.nrows; r += kLmEpiWarps * 32)
        if (s_key[r] != 0ull) atomicMax(&keys[r], s_key[r]);
    }
  }
  tc::fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc::fence_after();
    tc::dealloc(tmem, 512);
  }
}

// One CTA per sequence: each row's argmax from its key, then the greedy rule of the mode.
__global__ void __launch_bounds__(256) lmhead_finalize(const __grid_constant__ LmheadParams p) {
  __shared__ int s_a[kLmMaxNodes];
  __shared__ int32_t tok[kLmMaxNodes];  // the sequence's node or draft tokens, staged by all threads
  const int b = blockIdx.x;
  const bool tree = p.mode == SPEC_SAMPLE_TREE_GREEDY;
  const int nt = tree ? p.R : p.R - 1;  // tokens to check: node tokens 1..N-1, or drafts 0..gamma-1
  // the tokens are inputs of the call, not of the GEMM: loaded before the wait
  for (int i = threadIdx.x; i < nt; i += blockDim.x) tok[i] = p.tok[(int64_t)b * p.tok_sb + i];
  pdl_wait();  // the GEMM's keys
  const unsigned long long* keys = reinterpret_cast<const unsigned long long*>(p.rec);
  for (int r = threadIdx.x; r < p.R; r += blockDim.x) s_a[r] = lm_key_id(__ldcg(keys + (int64_t)b * p.R + r));
  __syncthreads();
  if (threadIdx.x != 0) return;
  int32_t* out = p.out_tok + (int64_t)b * p.out_cols;
  int32_t* nodes = p.out_nodes ? p.out_nodes + (int64_t)b * p.out_cols : nullptr;
  bool bad = false;
  for (int i = tree ? 1 : 0; i < nt; ++i) bad |= tok[i] < 0 || tok[i] >= p.V;
  for (int c = 0; c < p.out_cols; ++c) {
    out[c] = -1;
    if (nodes) nodes[c] = -1;
  }
  if (bad) {
    p.out_nacc[b] = -1;
    atomicOr(p.status, (uint32_t)SPEC_STATUS_BAD_TOKEN);
    return;
  }
  if (!tree) {  // accept x_i while it equals the argmax of row i; then the argmax of row k
    int k = 0;
    while (k < p.R - 1 && tok[k] == s_a[k]) ++k;
    for (int i = 0; i < k; ++i) out[i] = tok[i];
    out[k] = s_a[k];
    p.out_nacc[b] = k;
    return;
  }
  // tree: node i accepted iff its parent is and its token is the parent row's argmax; the deepest
  // accepted node (ties to the smallest index), its path, then the argmax of its row
  unsigned long long acc = 1ull;
  int best = 0;
  for (int i = 1; i < p.R; ++i) {
    const int par = p.parent[i];
    if (((acc >> par) & 1ull) && tok[i] == s_a[par]) {
      acc |= 1ull << i;
      if (p.depth[i] > p.depth[best]) best = i;
    }
  }
  const int dd = p.depth[best];
  for (int j = best, k = dd - 1; j > 0; j = p.parent[j], --k) {
    out[k] = tok[j];
    if (nodes) nodes[k] = j;
  }
  out[dd] = s_a[best];
  p.out_nacc[b] = dd;
}

// The kernel's rings follow the parameters; they must be the layout's (the rings fit the
// dynamic shared memory it sizes, and each ring holds at least the copies of one group).
static bool lmhead_layout_matches(const LmLayout& L, const LmheadParams& p) {
  return L.w_stages == p.w_stages && L.h_stages == p.h_stages && L.kgroup == p.kgroup && L.wbox == p.wbox &&
         L.hbox == p.hbox && L.w_stages >= (L.kgroup + L.wbox - 1) / L.wbox &&
         L.h_stages >= (L.kgroup + L.hbox - 1) / L.hbox && L.w_stages <= kLmWStagesMax &&
         L.h_stages <= kLmHStagesMax;
}

size_t lmhead_workspace_bytes(int nrows) { return 256 + (size_t)nrows * sizeof(unsigned long long); }

void lmhead_workspace_carve(void* ws, LmheadParams* p) {
  uint8_t* b = reinterpret_cast<uint8_t*>(ws);
  p->status = reinterpret_cast<uint32_t*>(b);
  p->rec = b + 256;
}

cudaError_t launch_lmhead(const LmheadParams& p, const CUtensorMap* tmW, const CUtensorMap* tmH, int num_sms,
                          cudaStream_t stream) {
  // the status word and the keys (0 lies below every real key) in one memset
  cudaError_t e = cudaMemsetAsync(p.status, 0, lmhead_workspace_bytes(p.nrows), stream);
  if (e != cudaSuccess) return e;
  const LmLayout L = lmhead_layout(p.npad);
  if (!lmhead_layout_matches(L, p)) return cudaErrorInvalidValue;
  // the limit is the largest layout's (a fixed value, so concurrent calls never race on it)
  e = ensure_dynamic_smem(reinterpret_cast<const void*>(lmhead_gemm<false>), kLmSmemCap - 2560);
  if (e != cudaSuccess) return e;
  const int grid = p.n_vtiles < num_sms ? p.n_vtiles : num_sms;
  lmhead_gemm<false><<<grid, kLmThreads, L.smem, stream>>>(*tmW, *tmH, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  return launch_dependent(lmhead_finalize, dim3(p.B), dim3(256), 0, stream, 0u, p);
}

cudaError_t launch_lmhead_logits(const LmheadParams& p, const CUtensorMap* tmW, const CUtensorMap* tmH, int num_sms,
                                 cudaStream_t stream) {
  const LmLayout L = lmhead_layout(p.npad);
  if (!lmhead_layout_matches(L, p) || !p.logits) return cudaErrorInvalidValue;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(lmhead_gemm<true>), kLmSmemCap - 2560);
  if (e != cudaSuccess) return e;
  const int grid = p.n_vtiles < num_sms ? p.n_vtiles : num_sms;
  lmhead_gemm<true><<<grid, kLmThreads, L.smem, stream>>>(*tmW, *tmH, p);
  return cudaGetLastError();
}

}  // namespace specv
