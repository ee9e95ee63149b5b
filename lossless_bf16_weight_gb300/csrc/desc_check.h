// Host-side check of a blob descriptor passed to an entry point.
#pragma once
#include "uw.h"

namespace uw {

// A descriptor as uw_blob_info fills it: consistent sizes, sections in order
// inside blob_bytes, a prefix code on the palette.  Every entry point that
// reads a blob refuses (UW_ERR_INVALID_ARG) one that is not.
bool desc_ok(const uw_desc &d);

}  // namespace uw
