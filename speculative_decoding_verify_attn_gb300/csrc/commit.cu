// The rollback step after verification: keep the K/V of the accepted tokens ("Speculative Decoding
// in LLM Serving Systems", Accepting and rejecting; "Guide to MagicDec", Implementation Step 3;
// "Speculative Decoding & Medusa" §4, the accepted path of a token tree).
//
// One thread-block cluster per sequence, CTA r of the cluster taking kv heads r, r + CS, ...:
// chain: the length drops to the accepted prefix, nothing moves.  Tree: for each of its heads a CTA
// first stages the path nodes' K/V rows in shared memory and only then writes them to their new
// positions (sources and destinations of different path nodes overlap: node j moves from
// kv_len - N + n_j to kv_len - N + 1 + j, and n_j >= j + 1), in 4-byte words.  Every CTA reads
// kv_len[b] first; after a cluster barrier, CTA 0 alone writes it.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "commit_internal.h"
#include "common.cuh"
#include "launch_cache.h"

namespace specv {

constexpr int kCommitThreads = 256;

__global__ void __launch_bounds__(kCommitThreads) commit_kernel(const __grid_constant__ CommitParams p) {
  extern __shared__ uint32_t s_rows[];  // [2][k][row words]: K rows, then V rows
  __shared__ int s_path[kCommitMaxNodes];
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  const int CS = (int)cl.num_blocks(), rank = (int)cl.block_rank();
  const int b = blockIdx.x / CS, tid = threadIdx.x;
  const int L = p.kv_len[b];
  const int k = p.num_accepted[b];
  int path_bad = 0;
  if (p.mode == SPEC_COMMIT_TREE && tid < p.nq - 1) {
    const int n = (tid < k && tid < p.path_cols) ? p.path_nodes[(int64_t)b * p.path_sb + tid] : 1;
    s_path[tid] = n;
    path_bad = tid < k && (n < 1 || n >= p.nq);
  }
  // every thread takes the same verdict (k and L are the same for the whole CTA)
  int bad = __syncthreads_or(path_bad) ? SPEC_STATUS_BAD_TOKEN : 0;
  if (k < 0 || k > p.nq - 1 || (p.mode == SPEC_COMMIT_TREE && k > p.path_cols)) bad |= SPEC_STATUS_BAD_TOKEN;
  if (L < p.nq || L > p.Lmax) bad |= SPEC_STATUS_BAD_KV_LEN;
  if (bad) {  // the same verdict in every CTA of the cluster: none of them writes anything
    if (tid == 0 && rank == 0) atomicOr(p.status, (uint32_t)bad);
    return;
  }
  const int base = L - p.nq;
  if (p.mode == SPEC_COMMIT_TREE && k > 0) {
    const int words = p.D * (p.bf16 ? 2 : 4) / 4;  // 4-byte words per row
    const int per = k * words;
    for (int g = rank; g < p.Hkv; g += CS) {
      const int64_t head = (int64_t)b * p.kv_sb + (int64_t)g * p.kv_sh;  // elements
      const uint32_t* ks = reinterpret_cast<const uint32_t*>(reinterpret_cast<const char*>(p.k) +
                                                             head * (p.bf16 ? 2 : 4));
      const uint32_t* vs = reinterpret_cast<const uint32_t*>(reinterpret_cast<const char*>(p.v) +
                                                             head * (p.bf16 ? 2 : 4));
      for (int i = tid; i < per; i += kCommitThreads) {
        const int j = i / words, w = i - j * words;
        const int64_t src = (int64_t)(base + s_path[j]) * words + w;
        s_rows[i] = ks[src];
        s_rows[per + i] = vs[src];
      }
      __syncthreads();
      uint32_t* kd = const_cast<uint32_t*>(ks);
      uint32_t* vd = const_cast<uint32_t*>(vs);
      for (int i = tid; i < per; i += kCommitThreads) {
        const int j = i / words, w = i - j * words;
        const int64_t dst = (int64_t)(base + 1 + j) * words + w;
        kd[dst] = s_rows[i];
        vd[dst] = s_rows[per + i];
      }
      __syncthreads();
    }
  }
  cl.sync();  // every CTA of the cluster has read kv_len[b]
  if (tid == 0 && rank == 0) p.kv_len[b] = base + 1 + k;
}

size_t commit_smem_bytes(int nq, int D, int bf16) {
  return 2 * (size_t)(nq - 1) * (size_t)D * (bf16 ? 2 : 4);
}

cudaError_t launch_commit(const CommitParams& p, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(p.status, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess) return e;
  const size_t smem = p.mode == SPEC_COMMIT_TREE ? commit_smem_bytes(p.nq, p.D, p.bf16) : 0;
  if (smem > 48 * 1024) {
    e = ensure_dynamic_smem(reinterpret_cast<const void*>(commit_kernel), (int)smem);
    if (e != cudaSuccess) return e;
  }
  // one CTA per kv head (at most 8 per sequence) in tree mode, one per sequence in chain mode
  const int cs = p.mode == SPEC_COMMIT_TREE ? (p.Hkv < 8 ? p.Hkv : 8) : 1;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)(p.B * cs), 1, 1);
  cfg.blockDim = dim3(kCommitThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, commit_kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace specv
