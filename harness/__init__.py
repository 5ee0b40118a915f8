"""Device set-up of synthetic workloads for the CUDA path (GPU tests and benchmark)."""

from .device import LayerDev, WorkloadDev, n_visible  # noqa: F401
