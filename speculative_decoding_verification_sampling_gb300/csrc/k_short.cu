// Verification with a draft defined on a per-sequence shortlist.
#include "sv_instantiate.cuh"

namespace sv {

KernelEntry entry_short(int tdt, bool probs)
{
    if (tdt == 0)
        return probs ? make_entry<F32, MODE_SHORT, true>() : make_entry<F32, MODE_SHORT, false>();
    return probs ? make_entry<BF16, MODE_SHORT, true>() : make_entry<BF16, MODE_SHORT, false>();
}

}  // namespace sv
