// Kernel instantiations: GBFFT_DEF_REAL(9) GBFFT_DEF_REAL(10).
#include "inst_defs.cuh"
#include "inst_entries.h"

GBFFT_DEF_REAL(9)
GBFFT_DEF_REAL(10)
