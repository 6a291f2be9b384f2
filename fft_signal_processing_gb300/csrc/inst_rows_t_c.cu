// Kernel instantiations: GBFFT_DEF_ROWS_T(11).
#include "inst_defs.cuh"
#include "inst_entries.h"

GBFFT_DEF_ROWS_T(11)
