// Prints the L-group choices of the launch-shape helpers for the shapes the
// tests pin (compiled and run by tests/test_host_logic.py; host code only).
#include <cstdint>
#include <cstdio>

#include "../selective_state_space_07_gb300/csrc/ssm_internal.h"

int main() {
    // forward: (CTAs per group, SMs, resident CTAs per SM, cap)
    const int64_t fw[][4] = {{256, 152, 3, 8}, {192, 152, 3, 10}, {32, 152, 3, 64}, {32, 152, 3, 4},
                             {1, 152, 3, 1}, {0, 152, 3, 5}, {228, 152, 3, 64}, {227, 152, 3, 64}};
    for (const auto& r : fw) std::printf("fwd %d\n", ssm::choose_groups_fwd(r[0], r[1], r[2], r[3]));
    // backward: (CTAs per group, resident CTA capacity, cap), aggregate price 0.15
    const int64_t bw[][3] = {{128, 304, 8}, {96, 304, 10}, {16, 304, 64}, {128, 304, 1}, {4096, 304, 64}};
    for (const auto& r : bw) std::printf("bwd %d\n", ssm::choose_groups(r[0], r[1], 0.15, r[2]));
    return 0;
}
