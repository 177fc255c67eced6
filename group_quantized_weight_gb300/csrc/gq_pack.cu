// Offline repack of canonical weight codes into the device layouts gq_gemm streams.
//
// W4 ("GPU Kernel 工程（09）：量化与融合 kernel", section 3.3 item 1, and the interleaved nibble
// order required by the magic-number decode of section 2.4):
//   packed[t][c][lane][word j], t = 16-column tile, c = 64-k chunk, j = 16-k step in the
//   chunk.  Word j of lane L holds the eight codes lane L needs as the A operand of one
//   m16n8k16 tensor-core MMA whose rows are output columns n and whose columns are k:
//     pair i (i = 0..3) = rows r = L/4 + 8*(i & 1), k = 16j + 2*(L%4) + 8*(i >> 1) + {0,1}
//   with the first k of the pair at bits 4i..4i+3 and the second at bits 4i+16..4i+19,
//   so that (word >> 4i) & 0x000F000F leaves the two codes in the low bits of the two
//   16-bit halves, ready for the BF16 magic 0x4300.
// W4 fused gate+up (GQ_GATE_UP): tile t holds gate columns 8t .. 8t+7 as rows 0-7 and up
// columns N/2 + 8t .. as rows 8-15, so one lane's MMA results hold a gate column and its up
// column side by side.
// W8: 64-column blocks, each with its K/16 chunk rows contiguous: the 16 bytes at chunk row c
// of column n hold codes[16c + b][n], b = 0..15, so that a warp streaming one block's k range
// reads one contiguous run of memory.
#include "gq_internal.h"

namespace gq {

__global__ void pack_w4_kernel(int K, int N, const uint32_t *__restrict__ codes,
                               uint32_t *__restrict__ packed, size_t total_words, int gate_up) {
  const int nchunks = K / kChunkK;
  for (size_t o = blockIdx.x * (size_t)blockDim.x + threadIdx.x; o < total_words;
       o += (size_t)gridDim.x * blockDim.x) {
    const int j = (int)(o & 3);
    const int lane = (int)((o >> 2) & 31);
    const size_t tc = o >> 7;                  // tile * nchunks + chunk
    const int c = (int)(tc % nchunks);
    const int t = (int)(tc / nchunks);
    uint32_t word = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = (lane >> 2) + 8 * (i & 1);
      // fused gate+up: tile t holds gate columns 8t .. 8t+7 (rows 0-7) and the matching up
      // columns F + 8t .. (rows 8-15), F = N / 2
      const int n = gate_up ? (r < 8 ? 8 * t + r : N / 2 + 8 * t + r - 8) : t * kTileN + r;
      const int k = c * kChunkK + 16 * j + 2 * (lane & 3) + 8 * (i >> 1);   // even
      uint32_t lo = 0, hi = 0;
      if (n < N) {
        const uint32_t src = codes[(size_t)(k >> 3) * N + n];  // holds k and k + 1
        lo = (src >> (4 * (k & 7))) & 0xFu;
        hi = (src >> (4 * ((k + 1) & 7))) & 0xFu;
      }
      word |= lo << (4 * i);
      word |= hi << (4 * i + 16);
    }
    packed[o] = word;
  }
}

// gate_up: block b holds gate columns 32b .. 32b + 31 then up columns N/2 + 32b .. + 31 (the
// canonical column of packed column n)
__global__ void pack_w8_kernel(int K, int N, const int8_t *__restrict__ codes,
                               uint8_t *__restrict__ packed, size_t total_vecs, bool gate_up) {
  const size_t per_block = (size_t)(kColBlock8 / kChunkK8) * K;   // 16-byte vectors
  for (size_t o = blockIdx.x * (size_t)blockDim.x + threadIdx.x; o < total_vecs;
       o += (size_t)gridDim.x * blockDim.x) {
    const int b = (int)(o / per_block);
    const size_t rem = o - (size_t)b * per_block;
    const int wb = N - b * kColBlock8 < kColBlock8 ? N - b * kColBlock8 : kColBlock8;
    const size_t c = rem / wb;
    const int j = (int)(rem - c * wb), n = b * kColBlock8 + j;
    const int src = !gate_up ? n : j < 32 ? 32 * b + j : N / 2 + 32 * b + (j - 32);
    uint32_t w[4] = {0, 0, 0, 0};
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const uint32_t v = (uint8_t)codes[(c * 16 + e) * (size_t)N + src];
      w[e >> 2] |= v << (8 * (e & 3));
    }
    reinterpret_cast<uint4 *>(packed)[o] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

static int grid_for(size_t work, int threads) {
  size_t b = (work + threads - 1) / threads;
  if (b > 65535u * 8u) b = 65535u * 8u;
  return (int)(b ? b : 1);
}

cudaError_t launch_pack_w4(int K, int N, const uint32_t *codes, uint32_t *packed, bool gate_up,
                           cudaStream_t s) {
  const size_t tiles = (size_t)(N + kTileN - 1) / kTileN;
  const size_t total = tiles * (size_t)(K / kChunkK) * 128;
  pack_w4_kernel<<<grid_for(total, 256), 256, 0, s>>>(K, N, codes, packed, total,
                                                      gate_up ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_pack_w8(int K, int N, const int8_t *codes, uint8_t *packed, bool gate_up,
                           cudaStream_t s) {
  const size_t total = (size_t)(K / kChunkK8) * N;
  pack_w8_kernel<<<grid_for(total, 256), 256, 0, s>>>(K, N, codes, packed, total, gate_up);
  return cudaGetLastError();
}

}  // namespace gq
