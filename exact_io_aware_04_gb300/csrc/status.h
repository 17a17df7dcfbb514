// status.h -- status codes shared by host and device code of libattn.
#pragma once

#include "../../include/attn.h"
