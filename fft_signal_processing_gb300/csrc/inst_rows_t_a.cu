// Kernel instantiations: GBFFT_DEF_ROWS_T(8) GBFFT_DEF_ROWS_T(9).
#include "inst_defs.cuh"
#include "inst_entries.h"

GBFFT_DEF_ROWS_T(8)
GBFFT_DEF_ROWS_T(9)
