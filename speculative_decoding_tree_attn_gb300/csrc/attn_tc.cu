// Placeholder: the tcgen05 kernel is not built yet.
#include "attn_tc.h"

namespace tv {
bool tc_supported(const DeviceInfo&, int, int, int, int) { return false; }
int tc_rows_per_unit(int rows) { return rows <= 128 ? 128 : 256; }
int launch_attn_tc(const AttnParams&, cudaStream_t) { return fail(TV_ERR_UNSUPPORTED, "tcgen05 kernel not built"); }
}  // namespace tv
