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

// 4-D descriptor over state planes [nplanes][4096 rows r = m*64 + n][64 columns] (16-bit):
// one box is the 64 rows (m = 0..63, n fixed) x 64 columns of one plane, i.e. the slice
// {S[(m, n), :]} for a fixed second key index n, landing as a [m][column] tile.
bool make_tmap_state_slices(CUtensorMap* map, const void* base, uint64_t nplanes);

// Reads (and optionally clears) the device status word of the current device.
int read_tc_status(bool clear);

// Device address of the status word on the current device (looked up once per device);
// nullptr on failure.
int* tc_status_ptr();

}  // namespace tm2
