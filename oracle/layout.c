/*
 * layout.c -- oracle: the blocked (swizzled) layout of block scales that
 * Blackwell block-scaled matrix multiplies read.  Test infrastructure only
 * (see fp4_oracle.h).
 *
 * [fp4-train] "Scope": the NVFP4 tensor-core matmul hands its e4m3 block
 * scales to the hardware after swizzling them into the layout that
 * torch._scaled_mm consumes.  The page names the layout but does not spell it
 * out; it is written here from the public description of the tensor cores'
 * block-scale-factor layout (the one cuBLASLt documents for its 16- and
 * 32-element block scaling modes):
 *
 *   - the scale matrix has one byte per block, [rows, cols] row-major
 *     (cols = K / 16 for NVFP4, K / 32 for MXFP4);
 *   - it is padded with zero bytes to [128 * ceil(rows / 128),
 *     4 * ceil(cols / 4)];
 *   - the padded matrix is cut into tiles of 128 rows x 4 columns, stored one
 *     after the other in row-major tile order (all tiles of the first 128
 *     rows, then the next 128 rows, ...), 512 bytes each;
 *   - inside a tile, the scale of tile row r (0..127) and tile column c
 *     (0..3) is byte 16 * (r mod 32) + 4 * floor(r / 32) + c.
 *
 * So the 512-byte tile is a [32][4][4] array indexed (r mod 32, r / 32, c).
 */
#include "fp4_oracle.h"

int64_t ora_blocked_scales_size(int64_t rows, int64_t cols) {
  if (rows < 0 || cols < 0) return -1;
  return 128 * ((rows + 127) / 128) * 4 * ((cols + 3) / 4);
}

/* Byte offset of the scale (r, c) of the padded matrix in the blocked
 * buffer; col_tiles = ceil(cols / 4). */
static int64_t blocked_offset(int64_t r, int64_t c, int64_t col_tiles) {
  int64_t tile = (r / 128) * col_tiles + c / 4;
  int64_t tr = r % 128, tc = c % 4;
  return 512 * tile + 16 * (tr % 32) + 4 * (tr / 32) + tc;
}

int ora_scales_to_blocked(const uint8_t* scales, int64_t rows, int64_t cols,
                          uint8_t* blocked) {
  if (rows < 0 || cols < 0) return 1;
  int64_t prow = 128 * ((rows + 127) / 128), pcol = 4 * ((cols + 3) / 4);
  int64_t col_tiles = pcol / 4;
  for (int64_t r = 0; r < prow; ++r)
    for (int64_t c = 0; c < pcol; ++c) {
      uint8_t v = (r < rows && c < cols) ? scales[r * cols + c] : 0;
      blocked[blocked_offset(r, c, col_tiles)] = v;
    }
  return 0;
}

int ora_scales_from_blocked(const uint8_t* blocked, int64_t rows, int64_t cols,
                            uint8_t* scales) {
  if (rows < 0 || cols < 0) return 1;
  int64_t col_tiles = (cols + 3) / 4;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c)
      scales[r * cols + c] = blocked[blocked_offset(r, c, col_tiles)];
  return 0;
}
