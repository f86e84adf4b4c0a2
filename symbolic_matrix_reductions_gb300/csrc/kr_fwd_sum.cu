// Sum reduction instances.
#define KR_FWD_LSE false
#define KR_FWD_LAUNCH launch_sum
#define KR_FWD_OCCUPANCY occupancy_sum
#include "kr_fwd.inc"
