// Absorbed-MLA decode (tcgen05 / TMEM path): not built yet.
#include "kernels.h"

namespace skd {
int launch_mla(const DecodeArgs &) { return SKD_EUNSUPPORTED; }
}  // namespace skd
