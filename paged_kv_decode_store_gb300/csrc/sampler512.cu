// The sampler kernel built with 512-thread CTAs, two per SM (sampler.cu
// chooses between the two builds for each launch).
#define PKVD_SAMP_THREADS 512
#define PKVD_SAMP_NS s512
#include "sampler_core.cuh"
