// OTIL selective latent transmit on P virtual ranks of one device (see otil.cu).
#pragma once
#include "common.cuh"

namespace dpp {

constexpr int kOtilMaxBlocks = 4096;  // sub-blocks per band
constexpr int kOtilMaxK = 256;        // sub-blocks sent per rank and step

// Host checks of dpp_otil_params (status code), and the sub-block count per band.
int otil_check(const dpp_otil_params* p);
int otil_blocks(const dpp_otil_params* p);

int launch_otil_step(const dpp_otil_params& p, const void* fresh, void* views, uint8_t* visited,
                     int32_t* sel, void* msg, cudaStream_t s);
int launch_otil_finalize(const dpp_otil_params& p, const void* fresh, void* views,
                         uint8_t* visited, int reset, cudaStream_t s);

}  // namespace dpp
