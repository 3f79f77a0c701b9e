// Greedy verification (T == 0): argmax of the target rows only.
#include "sv_instantiate.cuh"

namespace sv {

KernelEntry entry_greedy(int tdt)
{
    return tdt == 0 ? make_entry<F32, MODE_GREEDY, false>() : make_entry<BF16, MODE_GREEDY, false>();
}

}  // namespace sv
