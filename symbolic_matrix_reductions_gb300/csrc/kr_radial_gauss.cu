// Max / Min of the Gaussian, and its Sum for the block-sparse mode (the dense Sum has its own kernels).
#define KR_RADIAL_KT KT_GAUSS
#define KR_RADIAL_SUM 1
#define KR_RADIAL_LAUNCH launch_radial_gauss
#define KR_RADIAL_OCCUPANCY occupancy_radial_gauss
#include "kr_radial.inc"
