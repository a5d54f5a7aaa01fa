// Scale repack: plain [L][rows][K/16] E4M3 bytes -> 128x4-atom layout.
//
// The destination is the pre-permuted scale tensor [32, 4, rest_m, 4, rest_k,
// L] of kernelbot nvfp4-gemv submission 103289 (`permuted_to_blocked`),
// stored L-outermost so that permuting it to [rest_m, rest_k, 32, 4, 4] is the
// blocked order that submission 69953's `to_blocked_batch` builds: byte
// (m, kb) of batch l goes to
//   ((l*rest_m + m/128)*rest_k + kb/4)*512 + (m%32)*16 + ((m/32)%4)*4 + kb%4.
// Rows past `rows` in the last 128-row block are written as 0x00.
//
// Each tile is one 128-row block by kTileCols atom columns (4 scale bytes per
// row each).  The tile's source words are read row by row (coalesced, 4-byte
// loads since plain rows are only 4-byte aligned), staged in shared memory,
// and written back as whole 512-byte atoms with 16-byte stores.  The grid is
// sized to the SMs and strides over tiles.
//
// When every plain row starts on a 16-byte boundary (K % 256 == 0 and a
// 16-byte aligned source) a register transpose does the same permutation with
// no shared memory: one thread reads 16 bytes (4 atom columns) of rows i,
// 32+i, 64+i, 96+i of a 128-row block and writes position i of those 4 atoms.
#include <cstdint>

#include "internal.h"

namespace nvfp4 {

namespace {

constexpr int kRepackThreads = 256;
constexpr int kTileCols = 16;               // atom columns per tile (64 scale bytes per row)
constexpr int kTileWords = 128 * kTileCols; // 4-byte words per tile
constexpr int kPitch = kTileCols + 1;       // odd pitch: conflict-free column gathers

__global__ void __launch_bounds__(kRepackThreads)
    repack_scales_kernel(const uint32_t* __restrict__ src, uint4* __restrict__ dst, int64_t rows,
                         int32_t rest_m, int32_t rest_k, int64_t tiles) {
  __shared__ uint32_t tile[128 * kPitch];
  const int64_t col_tiles = (rest_k + kTileCols - 1) / kTileCols;
  const int64_t row_words = rest_k;  // K/16 bytes per plain row = rest_k 4-byte words
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
    const int64_t ct = t % col_tiles;
    const int64_t mb = (t / col_tiles) % rest_m;
    const int64_t l = t / (col_tiles * rest_m);
    const int64_t col0 = ct * kTileCols;
    const int ncols = (int)(rest_k - col0 < kTileCols ? rest_k - col0 : kTileCols);
#pragma unroll
    for (int w = threadIdx.x; w < kTileWords; w += kRepackThreads) {
      const int r = w / kTileCols, cidx = w % kTileCols;
      const int64_t m = mb * 128 + r;
      uint32_t v = 0;
      if (m < rows && cidx < ncols) v = src[(l * rows + m) * row_words + col0 + cidx];
      tile[r * kPitch + cidx] = v;
    }
    __syncthreads();
    // one 16-byte output vector = rows i, 32+i, 64+i, 96+i of one atom column
    for (int v = threadIdx.x; v < 32 * kTileCols; v += kRepackThreads) {
      const int cidx = v / 32, i = v % 32;
      if (cidx < ncols) {
        uint4 o;
        o.x = tile[(i)*kPitch + cidx];
        o.y = tile[(32 + i) * kPitch + cidx];
        o.z = tile[(64 + i) * kPitch + cidx];
        o.w = tile[(96 + i) * kPitch + cidx];
        dst[((l * rest_m + mb) * rest_k + col0 + cidx) * 32 + i] = o;
      }
    }
    __syncthreads();
  }
}

constexpr int kVecThreads = 128;

// Thread u: lanes cover 4 consecutive 16-byte columns of 8 consecutive rows
// (64 contiguous source bytes per row, 128 contiguous destination bytes per
// atom and store); warps then step over column groups, the 4 row groups
// i/8 and finally the (l, 128-row block) pairs.
__global__ void __launch_bounds__(kVecThreads)
    repack_scales_vec_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t rows,
                             int32_t rest_m, int32_t qw, int64_t units) {
  const int64_t u = (int64_t)blockIdx.x * kVecThreads + threadIdx.x;
  if (u >= units) return;
  const int32_t groups = (qw + 3) / 4;  // 4-column groups per row
  const int ql = (int)(u % 4), il = (int)((u / 4) % 8);
  const int64_t w = u / 32;
  const int32_t q = (int32_t)(w % groups) * 4 + ql;
  if (q >= qw) return;
  const int i = (int)((w / groups) % 4) * 8 + il;
  const int64_t blk = w / ((int64_t)groups * 4);  // l * rest_m + m / 128
  const int64_t l = blk / rest_m;
  const int64_t m0 = (blk - l * rest_m) * 128 + i;
  uint4 x[4];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const int64_t m = m0 + 32 * g;
    x[g] = m < rows ? src[(l * rows + m) * qw + q] : make_uint4(0, 0, 0, 0);
  }
  uint4* out = dst + (blk * (int64_t)qw * 4 + (int64_t)q * 4) * 32 + i;
  out[0] = make_uint4(x[0].x, x[1].x, x[2].x, x[3].x);
  out[32] = make_uint4(x[0].y, x[1].y, x[2].y, x[3].y);
  out[64] = make_uint4(x[0].z, x[1].z, x[2].z, x[3].z);
  out[96] = make_uint4(x[0].w, x[1].w, x[2].w, x[3].w);
}

// Any K % 16 == 0 (plain rows K/16 bytes long, not always 4-byte aligned):
// thread w writes the w-th 4-byte word of the output, gathering its 4 scale
// bytes (blocks past K/16 and rows past `rows` are 0x00).
__global__ void __launch_bounds__(kRepackThreads)
    repack_scales_bytes_kernel(const uint8_t* __restrict__ src, uint32_t* __restrict__ dst,
                               int64_t rows, int64_t blocks, int32_t rest_m, int32_t rest_k,
                               int64_t words) {
  for (int64_t w = (int64_t)blockIdx.x * kRepackThreads + threadIdx.x; w < words;
       w += (int64_t)gridDim.x * kRepackThreads) {
    const int64_t atom = w / 128;              // (l*rest_m + m/128)*rest_k + kc
    const int in_atom = (int)(w % 128);        // i*4 + g: row 32*g + i of the block
    const int i = in_atom / 4, g = in_atom % 4;
    const int64_t kc = atom % rest_k, blk = atom / rest_k;  // blk = l*rest_m + m/128
    const int64_t l = blk / rest_m;
    const int64_t m = (blk - l * rest_m) * 128 + 32 * g + i;
    uint32_t v = 0;
    if (m < rows) {
      const uint8_t* row = src + (l * rows + m) * blocks;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int64_t kb = 4 * kc + t;
        if (kb < blocks) v |= (uint32_t)row[kb] << (8 * t);
      }
    }
    dst[w] = v;
  }
}

}  // namespace

cudaError_t repack_ctas_per_sm(int* out) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, repack_scales_kernel, kRepackThreads,
                                                       0);
}

cudaError_t launch_repack(const uint8_t* src, uint8_t* dst, int64_t rows, int64_t K, int64_t L,
                          int64_t max_ctas, cudaStream_t stream) {
  const int32_t rest_m = (int32_t)((rows + 127) / 128);
  const int32_t rest_k = (int32_t)((K + 63) / 64);
  if (K % 64 != 0) {
    const int64_t words = L * rest_m * (int64_t)rest_k * 128;
    if (words == 0) return cudaSuccess;
    const int64_t cap = max_ctas > 0 ? max_ctas : 1;
    const int64_t need = (words + kRepackThreads - 1) / kRepackThreads;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(need < cap ? need : cap), 1, 1);
    cfg.blockDim = dim3(kRepackThreads, 1, 1);
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, repack_scales_bytes_kernel, src,
                              reinterpret_cast<uint32_t*>(dst), rows, K / 16, rest_m, rest_k,
                              words);
  }
  const int32_t qw = rest_k / 4;
  const int64_t units = L * rest_m * 32 * (int64_t)((qw + 3) / 4) * 4;
  if (rest_k % 4 == 0 && reinterpret_cast<uintptr_t>(src) % 16 == 0 &&
      units <= (int64_t)0x7fffffff * kVecThreads) {
    if (units == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((units + kVecThreads - 1) / kVecThreads), 1, 1);
    cfg.blockDim = dim3(kVecThreads, 1, 1);
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, repack_scales_vec_kernel, reinterpret_cast<const uint4*>(src),
                              reinterpret_cast<uint4*>(dst), rows, rest_m, qw, units);
  }
  const int64_t tiles = L * rest_m * ((rest_k + kTileCols - 1) / kTileCols);
  if (tiles == 0) return cudaSuccess;
  const int64_t cap = max_ctas > 0 ? max_ctas : 1;
  const int64_t grid = tiles < cap ? tiles : cap;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kRepackThreads, 1, 1);
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, repack_scales_kernel, reinterpret_cast<const uint32_t*>(src),
                            reinterpret_cast<uint4*>(dst), rows, rest_m, rest_k, tiles);
}

}  // namespace nvfp4
