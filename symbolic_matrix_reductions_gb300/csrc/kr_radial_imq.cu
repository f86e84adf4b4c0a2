// Sum and Max / Min with the inverse-multiquadric kernel.
#define KR_RADIAL_KT KT_IMQ
#define KR_RADIAL_SUM 1
#define KR_RADIAL_LAUNCH launch_radial_imq
#define KR_RADIAL_OCCUPANCY occupancy_radial_imq
#include "kr_radial.inc"
