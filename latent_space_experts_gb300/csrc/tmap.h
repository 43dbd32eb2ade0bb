// Host-side 2-D TMA tensor maps (cuTensorMapEncodeTiled through the runtime's driver entry
// point, looked up once per process).
#pragma once

#include <cuda.h>

namespace slmoe {

// A rows x cols tensor (cols innermost) with a row pitch of `pitch` elements, read in boxes
// of box_cols x box_rows; out-of-range elements read as zero.  elem_bytes must match dtype.
// Returns SLMOE_OK or SLMOE_ECUDA (with a message) when the encoding is refused.
int tmap_encode_2d(CUtensorMap *m, CUtensorMapDataType dtype, int elem_bytes, const void *base,
                   long long rows, long long cols, long long pitch, int box_cols, int box_rows,
                   CUtensorMapSwizzle swizzle);

// Packed FP4 codes: rows x K values, K / 2 bytes per row (K a multiple of 128, the base 32-byte
// aligned), read in boxes of 128 values x 128 rows with the 128-byte swizzle and expanded in
// shared memory to one byte per value (16 values in the first half of each 16-byte chunk).
int tmap_encode_fp4(CUtensorMap *m, const void *base, long long rows, long long K);

}  // namespace slmoe
