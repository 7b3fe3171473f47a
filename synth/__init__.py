"""Seeded synthetic 4D-STEM inputs (configuration + single-slice forward model).

Shared by the CPU oracle's tests and the CUDA path's tests and benchmark; holds
no reconstruction arithmetic.
"""
from . import configs, forward  # noqa: F401
