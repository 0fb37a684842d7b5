// Shape facts of a context, for host code outside the executor (checkpoints).
#pragma once
#include <stddef.h>

#include <vector>

#include "planner.h"

struct gpipe_ctx;

namespace gp {

// The context's layer dimensions, its layer count, the FFN width of every
// layer and the parameter count of the packing.
void describe_context(const gpipe_ctx* c, Dims* dm, int* L, std::vector<int>* ffn, size_t* params);
// Record a failure message on the context (what gpipe_last_error returns).
int context_fail(gpipe_ctx* c, int code, const char* msg);

}  // namespace gp
