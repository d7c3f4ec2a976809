"""GB300-native (sm_103a) LoGRA low-rank gradient sketching hot path.

The compute lives in ``_lib/liblogra.so`` (C ABI declared in
``include/logra.h``); this package is the thin Python binding over it plus the
host-side δ budget schedule.  Importing it loads the library and raises if it
has not been built.
"""

from ._binding import (  # noqa: F401
    LOGRA_DTYPE_BF16,
    LOGRA_DTYPE_FP32,
    LOGRA_PROJ_BF16,
    LOGRA_PROJ_FP32,
    LOGRA_PROJ_GAUSS_BF16,
    LOGRA_PROJ_GAUSS_FP32,
    LOGRA_PROJ_INT8_PM1,
    LOGRA_PROJ_SIGN_BF16,
    LograError,
    MergeGroupPlan,
    SketchGroupPlan,
    lib,
    logra_device_error,
    logra_kl_workspace_bytes,
    logra_last_error,
    logra_merge_group_plan,
    logra_merge_group_plan_bytes,
    logra_merge_update,
    logra_merge_update_group,
    logra_merge_update_proj,
    logra_predicted_kl,
    logra_predicted_kl_noalloc,
    logra_refreshed_seed,
    logra_self_test_wait_timeout,
    logra_regen_projection,
    logra_sketch_accumulate,
    logra_sketch_accumulate_group,
    logra_sketch_group_plan,
    logra_sketch_group_plan_bytes,
    logra_sketch_group_workspace_bytes,
    logra_sketch_accumulate_proj,
    logra_sketch_momentum,
    logra_sum_squares,
    logra_sketch_accumulate_shared_x,
    logra_sketch_accumulate_shared_x_proj,
    logra_sketch_shared_x_workspace_bytes,
    logra_sketch_splits,
    logra_sketch_workspace_bytes,
    logra_step_size,
    logra_step_size_device,
    logra_version,
    sketch_workspace,
)
from .schedule import delta_schedule  # noqa: F401
