// LogSumExp reduction instances.
#define KR_FWD_LSE true
#define KR_FWD_LAUNCH launch_lse
#define KR_FWD_OCCUPANCY occupancy_lse
#include "kr_fwd.inc"
