// qmm_internal.h -- facts about the current device shared by the library's
// translation units (not exported).
#pragma once

namespace qmm {

// SM count and opt-in shared memory per block of the current device, looked
// up once per device; false unless it is an sm_103 device.
bool device_facts(int* sms, int* smem_optin);

}  // namespace qmm
