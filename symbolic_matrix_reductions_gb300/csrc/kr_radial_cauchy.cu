// Sum and Max / Min with the cauchy kernel.
#define KR_RADIAL_KT KT_CAUCHY
#define KR_RADIAL_SUM 1
#define KR_RADIAL_LAUNCH launch_radial_cauchy
#define KR_RADIAL_OCCUPANCY occupancy_radial_cauchy
#include "kr_radial.inc"
