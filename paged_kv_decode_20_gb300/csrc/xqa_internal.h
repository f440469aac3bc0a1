// Library-internal helpers shared between the C ABI translation units.
#pragma once

namespace xqa {

// Sets the text that xqa_last_error() returns on the calling thread.
void set_last_error(const char* msg);

}  // namespace xqa
