// Kernel instantiations: GBFFT_DEF_BLUESTEIN(13) GBFFT_DEF_BLUESTEIN(14).
#include "inst_defs.cuh"
#include "inst_entries.h"

GBFFT_DEF_BLUESTEIN(13)
GBFFT_DEF_BLUESTEIN(14)
