// tm2_tc.h -- host helpers of the tensor-core kernels (internal to the library).
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace tm2 {

// 2-D bf16 TMA descriptor over a row-major [rows][cols] matrix (row pitch in elements),
// box of box_rows x 64 columns, 128-byte swizzle, zero fill outside the matrix.
bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                       uint64_t pitch_elems, uint32_t box_rows);

// 3-D bf16 TMA descriptor over a dense [heads][rows][cols] tensor (cols a multiple of 8),
// box of 1 head x box_rows rows x 64 columns, 128-byte swizzle; rows past the end of a head
// read as zero.
bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, uint64_t heads, uint64_t rows, uint64_t cols,
                       uint32_t box_rows);

// Tiled map over 16-bit data, `rank` <= 5 dimensions: dims[i] extents (dims[0] contiguous),
// strides[i - 1] the byte stride of dimension i (any order, multiples of 16), box[i] the box;
// 128-byte swizzle, box[0] = 64.  The box lands in shared memory dimension 0 fastest.
bool make_tmap_f16_nd(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                      const uint32_t* box);

// Block-packed states (TC_PACKED_ROWS rows per plane): four rows m' = 4 mq .. 4 mq + 3 of one
// 16 x 16 block, all its 16 columns n' (smem [m'][n'][col], 8 KB).  Coordinates
// (0, 0, 16 block + 4 mq, 2 chunk + plane).
bool make_tmap_state_packed_quads(CUtensorMap* map, const void* base, uint64_t nchunks);
// One whole block plane of the block-packed states as [256 rows][64] (32 KB), rows r = 16 m' + n'.
// Coordinates (0, 256 block, 2 chunk + plane).
bool make_tmap_state_packed_blocks(CUtensorMap* map, const void* base, uint64_t nchunks);
// Block-packed states seen the other way round: all 16 rows m' of one 16 x 16 block for four
// of its columns n' = 4 nq .. 4 nq + 3 (smem [n'][m'][col], 8 KB).  Coordinates
// (0, 0, 4 nq, 10 (2 chunk + plane) + block).
bool make_tmap_state_packed_tquads(CUtensorMap* map, const void* base, uint64_t nchunks);
// A run of nb consecutive packed blocks (one block row (bm, bm + i), i < nb), from each its
// rows m' = 4 mq .. 4 mq + 3 with all 16 columns n' (smem [block][m'][n'][col], nb x 8 KB).
// Coordinates (0, 0, 4 mq, first block, 2 chunk + plane).  nb = 1 .. 4.
bool make_tmap_state_packed_rowrun(CUtensorMap* map, const void* base, uint64_t nchunks, int nb);

// Reads (and optionally clears) the device status word of the current device.
int read_tc_status(bool clear);

// Device address of the status word on the current device (looked up once per device);
// nullptr on failure.
int* tc_status_ptr();

}  // namespace tm2
