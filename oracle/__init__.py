"""fp64 CPU oracle of the GDN mixer core: test infrastructure, never part of the product path."""
