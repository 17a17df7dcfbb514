// status.h -- status codes shared by host and device code of libattn.
#pragma once

#include "attn.h"  // include/attn.h (on the -I path)
