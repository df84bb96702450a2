// objective.h -- launch interface of the ACR token objective (objective.cu).
#pragma once
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace qurl {

// Workspace: kAcrMaxCtas rows of 8 doubles (per-CTA partials), then the ticket
// counter, which must be zero before a call and is left zero.
constexpr int kAcrMaxCtas = 1024;
constexpr size_t kAcrTicketOffset = static_cast<size_t>(kAcrMaxCtas) * 8 * sizeof(double);
constexpr size_t kAcrWorkspaceBytes = kAcrTicketOffset + 256;

int acr_grid(long long T, int num_sms);
cudaError_t launch_acr_objective(const float* lp, const float* lpp, const float* lpb, const float* adv,
                                 const uint8_t* mask, long long T, float eps, float C, int adaptive, float* term,
                                 float* dterm, double* stats, void* workspace, int num_sms, cudaStream_t st);

}  // namespace qurl
