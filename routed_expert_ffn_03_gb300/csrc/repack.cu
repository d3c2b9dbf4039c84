// repack.cu - boundary blob -> kernel layout of one expert record (device to device).
//
// The boundary format is the plain one documented in include/moe.h; the layout it is
// turned into is described in layout.h.  Both kernels compute each output word from
// its own position, so they read the blob in any order and write the record once.
#include "kernels.h"

namespace moe {

// int4: one thread per output u32 word of a matrix.
__global__ void repack_int4_kernel(const uint8_t* __restrict__ nib,
                                   const uint16_t* __restrict__ scales, int R, int K,
                                   uint32_t* __restrict__ dst, MatGeom g) {
  const size_t per_pair = (size_t)g.ngroup * (I4_PAIR_BLOCK / 4);
  const size_t nwords = (size_t)g.ntask * per_pair;
  const int KH = K / 2, NG = K / I4_GROUP;
  for (size_t w = (size_t)blockIdx.x * blockDim.x + threadIdx.x; w < nwords;
       w += (size_t)gridDim.x * blockDim.x) {
    const int task = (int)(w / per_pair);
    const size_t rem = w % per_pair;
    const int group = (int)(rem / (I4_PAIR_BLOCK / 4));
    const int in_pair = (int)(rem % (I4_PAIR_BLOCK / 4));
    const int tile = in_pair / (I4_BLOCK / 4);
    const int within = in_pair % (I4_BLOCK / 4);
    const int rbase = task * 32 + tile * 16;
    uint32_t v = 0;
    if (within < 256) {
      const int kc = within / 128, lane = (within / 4) % 32, j = within % 4;
      const int gq = lane >> 2, p = lane & 3;
      const int kb = group * I4_GROUP + (kc * 4 + j) * 16;
      const int r = rbase + gq, r8 = r + 8;
      auto nb = [&](int row, int k) -> uint32_t {
        if (row >= R) return 0u;
        const uint8_t b = nib[(size_t)row * KH + (k >> 1)];
        return (k & 1) ? (uint32_t)(b >> 4) : (uint32_t)(b & 15);
      };
      v = nb(r, kb + 2 * p) | (nb(r, kb + 2 * p + 1) << 16) | (nb(r8, kb + 2 * p) << 4) |
          (nb(r8, kb + 2 * p + 1) << 20) | (nb(r, kb + 2 * p + 8) << 8) |
          (nb(r, kb + 2 * p + 9) << 24) | (nb(r8, kb + 2 * p + 8) << 12) |
          (nb(r8, kb + 2 * p + 9) << 28);
    } else {
      const int gq = within - 256;
      const int r = rbase + gq, r8 = r + 8;
      const uint32_t s0 = r < R ? scales[(size_t)r * NG + group] : 0u;
      const uint32_t s1 = r8 < R ? scales[(size_t)r8 * NG + group] : 0u;
      v = s0 | (s1 << 16);
    }
    dst[w] = v;
  }
}

// RVQ: codebooks are copied; codes are permuted into lane streams.
__global__ void repack_rvq_kernel(const uint8_t* __restrict__ blob, int R, int K,
                                  uint32_t* __restrict__ dst, MatGeom g) {
  const uint8_t* codes = blob + RVQ_CB_BYTES;
  const int G = K / RVQ_GROUP;
  const size_t ncb = RVQ_CB_BYTES / 4;
  const size_t per_task = RVQ_TASK_BYTES / 4;  // 1536 words
  const size_t nwords = ncb + (size_t)g.nks * g.ntask * per_task;
  for (size_t w = (size_t)blockIdx.x * blockDim.x + threadIdx.x; w < nwords;
       w += (size_t)gridDim.x * blockDim.x) {
    if (w < ncb) {  // the blob's matrix blocks are only byte aligned
      const uint8_t* b = blob + 4 * w;
      dst[w] = (uint32_t)b[0] | ((uint32_t)b[1] << 8) | ((uint32_t)b[2] << 16) | ((uint32_t)b[3] << 24);
      continue;
    }
    const size_t c = w - ncb;
    const size_t st = c / per_task;
    const int within = (int)(c % per_task);
    const int ks = (int)(st / g.ntask), rb = (int)(st % g.ntask);
    const int wq = within / 128, lane = (within / 4) % 32, j = within % 4;
    const int wi = wq * 4 + j;           // word of the lane stream, 0..47
    const int row = rb * 32 + lane;
    uint32_t v = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int bp = 4 * wi + b;         // byte of the lane stream, 0..191
      const int i = bp / 3, s = bp % 3;  // position i carries group (lane ^ i)
      const int q = ks * RVQ_KS + (lane ^ i);
      uint32_t code = 0;
      if (row < R && q < G) code = codes[((size_t)row * G + q) * 3 + s];
      v |= code << (8 * b);
    }
    dst[w] = v;
  }
}

cudaError_t launch_repack(int wfmt, const uint8_t* blob, int H, int F, uint8_t* rec,
                          cudaStream_t stream) {
  const RecGeom rg = rec_geom(wfmt, H, F);
  size_t boff = 0;
  for (int m = 0; m < 3; ++m) {
    const MatGeom& g = rg.m[m];
    uint32_t* dst = reinterpret_cast<uint32_t*>(rec + rg.off[m]);
    const int threads = 256;
    const size_t nwords = g.bytes / 4;
    const int blocks = (int)std::min<size_t>((nwords + threads - 1) / threads, 4096);
    if (wfmt == WFMT_INT4) {
      const uint8_t* nib = blob + boff;
      const uint16_t* sc =
          reinterpret_cast<const uint16_t*>(blob + boff + (size_t)g.rows * g.K / 2);
      repack_int4_kernel<<<blocks, threads, 0, stream>>>(nib, sc, g.rows, g.K, dst, g);
    } else {
      repack_rvq_kernel<<<blocks, threads, 0, stream>>>(blob + boff, g.rows, g.K, dst, g);
    }
    boff += blob_matrix_bytes(wfmt, g.rows, g.K);
  }
  return cudaGetLastError();
}

}  // namespace moe
