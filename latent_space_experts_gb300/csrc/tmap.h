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

}  // namespace slmoe
