// mla_decode.cu -- placeholder until the MLA decode kernels land.
#include "kernels.h"

namespace gbattn {

size_t mla_workspace_bytes(int, int, int, int, int) { return 0; }

int launch_mla_decode(const void *, const void *, const void *, const void *, void *, float *, int,
                      int, int, int, int, float, void *, size_t, const LaunchEnv &,
                      std::string &err)
{
    err = "mla_decode: not built yet";
    return 2;
}

}  // namespace gbattn
