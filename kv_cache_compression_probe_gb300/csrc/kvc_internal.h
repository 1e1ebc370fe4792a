// Internal declarations shared by the translation units of libkvc.
#pragma once
#include <stddef.h>
#include "../../include/kvc.h"

namespace kvc {
size_t score_workspace_bytes(const kvc_params* p);
size_t select_workspace_bytes(const kvc_params* p);
size_t pack_workspace_bytes(const kvc_params* p);
size_t decode_workspace_bytes(const kvc_params* p);
size_t partition_workspace_bytes(const kvc_params* p);
}  // namespace kvc
