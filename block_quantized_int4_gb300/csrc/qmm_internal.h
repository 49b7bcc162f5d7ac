// qmm_internal.h -- facts about the current device shared by the library's
// translation units (not exported).
#pragma once

namespace qmm {

// SM count and opt-in shared memory per block of the current device, looked
// up once per device; false unless it is an sm_103 device.
bool device_facts(int* sms, int* smem_optin);

// Device address of the library's device error word (read and cleared by
// qmm_last_device_error), or null without an sm_103 device.
int* device_error_word();

}  // namespace qmm
