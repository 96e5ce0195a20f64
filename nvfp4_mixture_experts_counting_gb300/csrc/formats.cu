// Intermediate-axis slicing of expert banks held in other formats, on the
// device (a load-time step).
//
// Issue #62 "Offloaded MoE ignores tensor parallelism: TP=2 is a regression,
// and the fix is not expert parallelism", section "What it touches": a rank's
// part of gate_up [2I, H] is two disjoint row ranges (gate rows [i0, i0+I_loc)
// and up rows [I+i0, I+i0+I_loc)), its part of down [H, I] is a column range;
// I_loc must stay a multiple of the format's block size (128 for fp8_block,
// 32 for the fp4 scale blocks, 32 for q4_0); mxfp4 is stored transposed
// (blocks_t [K/2, N]), so its gate_up slice runs along N and its down slice
// along the rows of blocks_t and of its scales.
//
// Every case is a few rectangles of bytes (rows x byte columns) copied from
// each expert's arrays into the sliced arrays; one kernel copies all the
// rectangles of a call, in 16-byte pieces where the rectangle allows it.
#include <cuda_runtime.h>

#include "../../include/ftmoe.h"

namespace {

constexpr int kMaxRects = 8;

struct Rect {
  int arr;              // which array of the format (0..2)
  int64_t src_off;      // bytes from the expert's first byte of the source array
  int64_t src_pitch;    // bytes between source rows
  int64_t dst_off, dst_pitch;
  int64_t width;        // bytes per row
  int64_t rows;
};

struct SliceArgs {
  const unsigned char* src[3];
  unsigned char* dst[3];
  int64_t src_expert[3];  // bytes of one expert's source array
  int64_t dst_expert[3];
  Rect r[kMaxRects];
  int n_rects;
  int E;
};

// Grid: x over row chunks, y over rectangles, z over experts.
__global__ void __launch_bounds__(256) k_slice_rects(const __grid_constant__ SliceArgs a) {
  const Rect& R = a.r[blockIdx.y];
  const int e = blockIdx.z;
  const unsigned char* src = a.src[R.arr] + (int64_t)e * a.src_expert[R.arr] + R.src_off;
  unsigned char* dst = a.dst[R.arr] + (int64_t)e * a.dst_expert[R.arr] + R.dst_off;
  const bool v16 = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15) == 0 &&
                   (R.src_pitch & 15) == 0 && (R.dst_pitch & 15) == 0 && (R.width & 15) == 0;
  const int64_t unit = v16 ? 16 : 1;
  const int64_t per_row = R.width / unit, total = per_row * R.rows;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / per_row, c = i % per_row;
    if (v16)
      *reinterpret_cast<uint4*>(dst + row * R.dst_pitch + 16 * c) =
          __ldg(reinterpret_cast<const uint4*>(src + row * R.src_pitch + 16 * c));
    else
      dst[row * R.dst_pitch + c] = src[row * R.src_pitch + c];
  }
}

int block_of(int fmt) {
  switch (fmt) {
    case FTMOE_FMT_NVFP4: return 16;
    case FTMOE_FMT_FP8_BLOCK: return 128;
    case FTMOE_FMT_Q4_0: return 32;
    case FTMOE_FMT_MXFP4: return 32;
    default: return 0;
  }
}

// Two row ranges (gate, then up) of an array with `row_bytes` per row and
// `rows_per_i` rows per intermediate index (1, or 1/128 for tile rows).
void add_gate_up_rows(SliceArgs& a, int arr, int64_t row_bytes, int64_t I, int64_t i0, int64_t I_loc, int64_t div) {
  a.r[a.n_rects++] = {arr, (i0 / div) * row_bytes, row_bytes, 0, row_bytes, row_bytes, I_loc / div};
  a.r[a.n_rects++] = {arr, ((I + i0) / div) * row_bytes, row_bytes, (I_loc / div) * row_bytes, row_bytes,
                      row_bytes, I_loc / div};
}

}  // namespace

extern "C" int ftmoe_slice_format(int format, int matrix, int E, int H, int I, int i0, int I_loc,
                                  const void* const* src, void* const* dst, ftmoe_stream_t stream) {
  const int b = block_of(format);
  if (!b || (matrix != FTMOE_MAT_GATE_UP && matrix != FTMOE_MAT_DOWN) || E < 0 || H <= 0 || I <= 0 || !src || !dst)
    return FTMOE_ERR_INVALID_ARG;
  if (I_loc <= 0 || i0 < 0 || i0 + I_loc > I) return FTMOE_ERR_INVALID_ARG;
  if (i0 % b || I_loc % b || I % b) return FTMOE_ERR_ALIGNMENT;
  if (H % b) return FTMOE_ERR_ALIGNMENT;  // whole blocks along H too (gate_up rows are H long)
  if (E == 0) return FTMOE_OK;
  const int narr = format == FTMOE_FMT_NVFP4 ? 3 : (format == FTMOE_FMT_Q4_0 ? 1 : 2);
  SliceArgs a{};
  a.E = E;
  for (int i = 0; i < narr; ++i) {
    if (!src[i] || !dst[i]) return FTMOE_ERR_INVALID_ARG;
    a.src[i] = static_cast<const unsigned char*>(src[i]);
    a.dst[i] = static_cast<unsigned char*>(dst[i]);
  }
  const int64_t h = H, in = I, s0 = i0, w = I_loc;
  const int64_t ht = (h + 127) / 128;  // fp8_block tile rows of down
  if (matrix == FTMOE_MAT_GATE_UP) {
    // gate_up [2I, H]
    switch (format) {
      case FTMOE_FMT_NVFP4:
        add_gate_up_rows(a, 0, h / 2, in, s0, w, 1);
        add_gate_up_rows(a, 1, h / 16, in, s0, w, 1);
        add_gate_up_rows(a, 2, 4, in, s0, w, 1);
        a.src_expert[0] = 2 * in * (h / 2), a.src_expert[1] = 2 * in * (h / 16), a.src_expert[2] = 2 * in * 4;
        a.dst_expert[0] = 2 * w * (h / 2), a.dst_expert[1] = 2 * w * (h / 16), a.dst_expert[2] = 2 * w * 4;
        break;
      case FTMOE_FMT_FP8_BLOCK:
        add_gate_up_rows(a, 0, h, in, s0, w, 1);
        add_gate_up_rows(a, 1, ht * 4, in, s0, w, 128);
        a.src_expert[0] = 2 * in * h, a.src_expert[1] = (2 * in / 128) * ht * 4;
        a.dst_expert[0] = 2 * w * h, a.dst_expert[1] = (2 * w / 128) * ht * 4;
        break;
      case FTMOE_FMT_Q4_0:
        add_gate_up_rows(a, 0, h / 32 * 18, in, s0, w, 1);
        a.src_expert[0] = 2 * in * (h / 32 * 18);
        a.dst_expert[0] = 2 * w * (h / 32 * 18);
        break;
      case FTMOE_FMT_MXFP4:
        // blocks_t [H/2][2I] and scales_t [H/32][2I]: two column ranges each
        for (int arr = 0; arr < 2; ++arr) {
          const int64_t rows = arr == 0 ? h / 2 : h / 32;
          a.r[a.n_rects++] = {arr, s0, 2 * in, 0, 2 * w, w, rows};
          a.r[a.n_rects++] = {arr, in + s0, 2 * in, w, 2 * w, w, rows};
          a.src_expert[arr] = rows * 2 * in;
          a.dst_expert[arr] = rows * 2 * w;
        }
        break;
    }
  } else {
    // down [H, I]: a column range
    switch (format) {
      case FTMOE_FMT_NVFP4:
        a.r[a.n_rects++] = {0, s0 / 2, in / 2, 0, w / 2, w / 2, h};
        a.r[a.n_rects++] = {1, s0 / 16, in / 16, 0, w / 16, w / 16, h};
        a.r[a.n_rects++] = {2, 0, 4 * h, 0, 4 * h, 4 * h, 1};  // every row global
        a.src_expert[0] = h * (in / 2), a.src_expert[1] = h * (in / 16), a.src_expert[2] = 4 * h;
        a.dst_expert[0] = h * (w / 2), a.dst_expert[1] = h * (w / 16), a.dst_expert[2] = 4 * h;
        break;
      case FTMOE_FMT_FP8_BLOCK:
        a.r[a.n_rects++] = {0, s0, in, 0, w, w, h};
        a.r[a.n_rects++] = {1, s0 / 128 * 4, in / 128 * 4, 0, w / 128 * 4, w / 128 * 4, ht};
        a.src_expert[0] = h * in, a.src_expert[1] = ht * (in / 128) * 4;
        a.dst_expert[0] = h * w, a.dst_expert[1] = ht * (w / 128) * 4;
        break;
      case FTMOE_FMT_Q4_0:
        a.r[a.n_rects++] = {0, s0 / 32 * 18, in / 32 * 18, 0, w / 32 * 18, w / 32 * 18, h};
        a.src_expert[0] = h * (in / 32 * 18);
        a.dst_expert[0] = h * (w / 32 * 18);
        break;
      case FTMOE_FMT_MXFP4:
        // blocks_t [I/2][H] and scales_t [I/32][H]: a range of whole rows
        a.r[a.n_rects++] = {0, s0 / 2 * h, h, 0, h, (w / 2) * h, 1};
        a.r[a.n_rects++] = {1, s0 / 32 * h, h, 0, h, (w / 32) * h, 1};
        a.src_expert[0] = (in / 2) * h, a.src_expert[1] = (in / 32) * h;
        a.dst_expert[0] = (w / 2) * h, a.dst_expert[1] = (w / 32) * h;
        break;
    }
  }
  int64_t most = 0;
  for (int i = 0; i < a.n_rects; ++i) most = a.r[i].rows * a.r[i].width > most ? a.r[i].rows * a.r[i].width : most;
  int64_t gx = (most / 16 + 255) / 256;
  gx = gx < 1 ? 1 : (gx > 1024 ? 1024 : gx);
  if (E > 65535) return FTMOE_ERR_INVALID_ARG;
  k_slice_rects<<<dim3((unsigned)gx, a.n_rects, E), 256, 0, (cudaStream_t)stream>>>(a);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FTMOE_OK : FTMOE_ERR_CUDA;
}
