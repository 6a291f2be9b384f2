// Kernel instantiations: GBFFT_DEF_RPAIR(11..12).
#include "inst_defs.cuh"
#include "inst_entries.h"

GBFFT_DEF_RPAIR(11)
GBFFT_DEF_RPAIR(12)
