// Order-0 Huffman byte accounting of the stored codes (kvtc_cache page,
// module docstring "Byte accounting" and KVTCKVCache.entropy_coding_gain).
// The coder is not on the hot path: a histogram kernel counts, per slot and
// packed position, how often each code value occurs in the store; the host
// then builds each kept component's Huffman code lengths from its counts and
// adds up the bytes, falling back to fixed width per slot where Huffman does
// not pay for itself.
#include <algorithm>
#include <cstdint>
#include <queue>
#include <vector>

#include "kvc_internal.h"

namespace kvc {

namespace {

constexpr int kHistThreads = 256;
constexpr int kHistRows = 128;          // rows staged per pass
constexpr int kMaxSmemBins = 16384;     // compact bins kept in shared memory

// Grid (slot, token span).  counts: [n_slots][NC][256], NC the layer's
// chunk-aligned positions; only the first 2^w entries of a position are used.
__global__ void __launch_bounds__(kHistThreads)
    code_histogram_kernel(const Params p, uint32_t* counts, int NC, int64_t S, int64_t span) {
  extern __shared__ __align__(16) unsigned char sm[];
  __shared__ uint32_t ch[32];    // chunk entries: first byte | width << 16 | (codes-1) << 20 | valid << 31
  __shared__ int binoff[257];    // compact bin offset of each position (+ total)
  const int slot = blockIdx.x, tid = threadIdx.x;
  const int beta = p.basis_of[slot];
  const int P = p.P[beta];
  if (tid < 32) {
    uint32_t e = 0u;
    int nch = 0;
    for (int s = 0; s < kMaxSeg; ++s) {
      const int32_t* sg = p.seg + ((size_t)beta * kMaxSeg + s) * 4;
      if (!sg[3]) break;
      const int n = (sg[3] + 7) / 8;
      if (tid < nch + n && !e) {
        const int ci = tid - nch, nc = min(8, sg[3] - ci * 8);
        e = (uint32_t)(sg[0] + sg[1] * ci) | ((uint32_t)sg[1] << 16) | ((uint32_t)(nc - 1) << 20) |
            (1u << 31);
      }
      nch += n;
    }
    ch[tid] = e;
  }
  __syncthreads();
  if (tid == 0) {
    int off = 0;
    for (int j = 0; j < NC; ++j) {
      const uint32_t e = ch[j >> 3];
      binoff[j] = off;
      if ((e >> 31) && (j & 7) <= (int)((e >> 20) & 7u)) off += 1 << ((e >> 16) & 0xfu);
    }
    binoff[NC] = off;
  }
  __syncthreads();
  const int nbins = binoff[NC];
  const bool in_smem = nbins <= kMaxSmemBins;
  uint32_t* bins = reinterpret_cast<uint32_t*>(sm);
  unsigned char* rows = sm + (in_smem ? (size_t)kMaxSmemBins * 4 : 0);
  if (in_smem)
    for (int i = tid; i < nbins; i += kHistThreads) bins[i] = 0u;
  uint32_t* gcount = counts + (size_t)slot * NC * 256;
  const unsigned char* src = p.store + p.pay_off[slot];
  const int64_t t0 = (int64_t)blockIdx.y * span, t1 = min(S, t0 + span);
  for (int64_t tb = t0; tb < t1; tb += kHistRows) {
    const int nrow = (int)min((int64_t)kHistRows, t1 - tb);
    __syncthreads();  // the previous pass is done with the staged rows
    // rows tb .. tb + nrow - 1: a 16-byte aligned run (tb is a multiple of 128)
    const int nv = (nrow * P + 15) >> 4;
    for (int i = tid; i < nv; i += kHistThreads)
      reinterpret_cast<uint4*>(rows)[i] = reinterpret_cast<const uint4*>(src + tb * P)[i];
    __syncthreads();
    for (int item = tid; item < nrow * 32; item += kHistThreads) {
      const int t = item >> 5, c = item & 31;
      const uint32_t e = ch[c];
      if (!(e >> 31)) continue;
      const int w = (int)((e >> 16) & 0xfu), nc = (int)((e >> 20) & 7u) + 1;
      const int a = t * P + (int)(e & 0xffffu);
      uint64_t bits = 0;
      for (int b = 0; b < w; ++b) bits |= (uint64_t)rows[a + b] << (8 * b);
      for (int k = 0; k < nc; ++k) {
        const uint32_t code = (uint32_t)(bits >> (w * k)) & ((1u << w) - 1u);
        const int j = 8 * c + k;
        if (in_smem) atomicAdd(&bins[binoff[j] + code], 1u);
        else atomicAdd(&gcount[(size_t)j * 256 + code], 1u);
      }
    }
  }
  __syncthreads();
  if (in_smem)
    for (int j = 0; j < NC; ++j) {
      const int n = binoff[j + 1] - binoff[j];
      for (int v = tid; v < n; v += kHistThreads) {
        const uint32_t c = bins[binoff[j] + v];
        if (c) atomicAdd(&gcount[(size_t)j * 256 + v], c);
      }
    }
}

}  // namespace

size_t histogram_bytes(int n_slots, int NC) { return (size_t)n_slots * NC * 256 * 4; }

cudaError_t launch_code_histogram(const Params& p, uint32_t* counts, int NC, int64_t S,
                                  cudaStream_t s, int* nk) {
  cudaError_t e = cudaMemsetAsync(counts, 0, histogram_bytes(p.n_slots, NC), s);
  if (e != cudaSuccess || S == 0) return e;
  const int64_t span = 8192;  // a multiple of the staged rows
  const size_t smem = (size_t)kMaxSmemBins * 4 + (size_t)kHistRows * 256 + 16;
  e = cudaFuncSetAttribute(code_histogram_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)p.n_slots, (unsigned)((S + span - 1) / span));
  code_histogram_kernel<<<grid, kHistThreads, smem, s>>>(p, counts, NC, S, span);
  ++*nk;
  return cudaGetLastError();
}

// Code lengths of an order-0 Huffman code for `counts` (0 for unused
// symbols; a lone symbol gets one bit): repeatedly merge the two lightest
// nodes, each merge adding one bit to every symbol below them.
std::vector<int> huffman_code_lengths(const uint32_t* counts, int n) {
  std::vector<int> len(n, 0);
  struct Node {
    uint64_t w;
    int id;
  };
  auto heavier = [](const Node& a, const Node& b) { return a.w > b.w || (a.w == b.w && a.id > b.id); };
  std::priority_queue<Node, std::vector<Node>, decltype(heavier)> pq(heavier);
  std::vector<std::vector<int>> members;
  for (int i = 0; i < n; ++i)
    if (counts[i]) {
      members.push_back({i});
      pq.push(Node{counts[i], (int)members.size() - 1});
    }
  if (members.size() == 1) {
    len[members[0][0]] = 1;
    return len;
  }
  while (pq.size() > 1) {
    const Node a = pq.top();
    pq.pop();
    const Node b = pq.top();
    pq.pop();
    std::vector<int> m = members[a.id];
    m.insert(m.end(), members[b.id].begin(), members[b.id].end());
    for (int i : m) ++len[i];
    members.push_back(std::move(m));
    pq.push(Node{a.w + b.w, (int)members.size() - 1});
  }
  return len;
}

}  // namespace kvc
