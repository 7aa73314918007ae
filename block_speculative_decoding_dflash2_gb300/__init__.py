"""DFlash2 block-parallel draft step for GB300 (sm_103a).

The compute path is the C-ABI library ``libdflash2.so`` (hand-written CUDA,
declared in ``include/dflash2.h``); ``binding`` marshals torch tensors into
its entry points.  ``runner`` holds a small host-side helper that owns the
device buffers of a batch (cache, block table, workspace) and calls the
entry points in order.
"""

from . import binding  # noqa: F401
from .binding import (BF16, F32, DFlash2Error, dflash2_append_context,  # noqa: F401
                      dflash2_draft_step, dflash2_read_device_status, dflash2_select_path,
                      dflash2_status_string, dflash2_validate_config, dflash2_verify_accept,
                      dflash2_version, dflash2_workspace_size)
