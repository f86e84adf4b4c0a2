// Sum and Max / Min with the laplace kernel.
#define KR_RADIAL_KT KT_LAPLACE
#define KR_RADIAL_SUM 1
#define KR_RADIAL_LAUNCH launch_radial_laplace
#define KR_RADIAL_OCCUPANCY occupancy_radial_laplace
#include "kr_radial.inc"
